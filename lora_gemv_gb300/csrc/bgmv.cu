// Plan-free BGMV: shrink and expand_slice with the tokens in their natural
// order, each token's adapter read straight from the index array.
//
// Pages: vLLM PR #15655 summary list (the LoRA kernel split into a shrink and
// an expand variant; blocks without work skipped; a mask-free path when one
// adapter serves every token); vLLM PR #11579 (bgmv_shrink and
// bgmv_expand(_slice), the fp32 rank buffer between them, split-K shrink
// whose partials are added, add_inputs); Punica issue #17 (BGMV: every input
// may use its own adapter).
//
// Design (GB300).  For a decode batch served by a few adapters the grouping
// step (a sort, then a plan read ahead of every operand) costs more than the
// contraction itself.  These kernels skip it: a block of 128 consecutive
// tokens (the MMA's M = 128 TMEM lanes) is contracted against every adapter's
// weights at once on the tcgen05 tensor cores, and each token lane keeps its
// own adapter's part.
//  - shrink: D[128, rows] = X[128, H] . A[rows, H]^T, rows = the adapters'
//    stacked A rows of this CTA's share (all adapters, a few, or a column
//    range of one).  X and A are staged by TMA (128-byte swizzle) through a
//    ring of stages fed by one producer thread, one thread issues the MMAs,
//    and H is split over a thread-block cluster.  Each token lane reads its
//    adapter's columns from TMEM and sends them to the CTA owning that token
//    row (st.async into its shared memory, counted on its mbarrier); owners
//    sum the cluster's partials in rank order (deterministic) and write y.
//  - expand: out[128, cols] (+)= Y_ext . B_ext^T, where Y_ext[t] holds
//    token t's y in its adapter's block of K = L * r (zeros elsewhere) and
//    B_ext stacks the adapters' B rows along K.  Adapters without a token in
//    the block are skipped (no loads, no MMA).  The out tile is staged by TMA
//    before the kernel waits for the shrink; y enters the tensor cores as a
//    hi + lo pair of the weight type after a per-row power-of-two scaling.
// The extra tensor-core work (up to L times the grouped contraction) stays
// far below the tensor ridge; what the design saves is the grouping launch
// and a dependent plan read in every operator.
#include <cudaTypedefs.h>
#include <string.h>

#include <algorithm>
#include <mutex>
#include <type_traits>

#include "common.cuh"
#include "fma_expand.cuh"
#include "frag.cuh"
#include "kernels.h"

namespace lora {
namespace {

constexpr int kBT = 128;        // tokens per block: MMA M and TMEM lanes
constexpr int kBThreads = 128;  // 4 warps, one TMEM lane quadrant each
constexpr int kBox = 64;        // K elements (128 bytes) per TMA box row
constexpr int kMaxStages = 4;
constexpr int kMaxCw = 64;      // y columns one shrink CTA produces, at most
constexpr int kShrinkSmemCap = 112 * 1024;  // keeps two shrink CTAs per SM

// 2-D fp16/bf16 tensor maps: make_tensor_map_2d (tmap.cu), boxes of
// box_rows x kBox columns.
cudaError_t make_map(CUtensorMap *m, lora_dtype_t dt, const void *base, uint64_t rows,
                     uint64_t cols, uint64_t ld, uint32_t box_rows) {
    return make_tensor_map_2d(m, dt, base, rows, cols, ld, box_rows);
}


// ------------------------------------------------------------------ shrink
// One launch's split, chosen on the host.  CTA (kc, block, z): K range
// [kc * kc_len, ...), tokens [128 * block, ...), and of the y columns the
// adapters [l_first, l_first + zk) x columns [c0, c0 + cw) with
// l_first = (z / zc) * zk and c0 = (z % zc) * cw: either whole adapters
// (zc = 1, cw = W = S * R) or one adapter's column range (zk = 1).
struct ShrinkSplit {
    int kc_len;  // K elements per CTA, a multiple of 64
    int nst;     // stages in the ring
    int zk, zc, cw;
    int n_mma;   // MMA N: A rows staged per stage (multiple of 16, <= 256)
    int tcols;   // TMEM columns allocated
};

template <typename E>
__global__ void __launch_bounds__(kBThreads)
bgmv_shrink_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_a,
                   const BgmvShrinkArgs a, const ShrinkSplit p) {
    extern __shared__ __align__(16) unsigned char smem[];
    __shared__ uint64_t s_full[kMaxStages], s_empty[kMaxStages], s_done, s_recv;
    __shared__ uint32_t s_tmem;
    __shared__ int s_l[kBT];
    const int tid = threadIdx.x, warp = tid >> 5;
    const int kc = (int)cluster_rank(), C = gridDim.x;
    const int t0 = blockIdx.y * kBT, z = blockIdx.z;
    const int W = a.S * a.R;
    const int l_first = (z / p.zc) * p.zk, c0 = (z % p.zc) * p.cw;
    const int l_count = min(p.zk, a.L - l_first);
    const int cw = min(p.cw, W - c0);  // a multiple of 8
    const int r0 = l_first * W + c0;   // first A row (of [L * W, H])
    const int k_begin = kc * p.kc_len;
    const int nk = (min(a.H, k_begin + p.kc_len) - k_begin + kBox - 1) / kBox;  // >= 1
    const int stage_bytes = kBT * 128 + p.n_mma * 128;
    const int RPO = kBT / C;  // token rows each cluster CTA finishes
    unsigned char *sm = smem + ((1024 - (smem_u32(smem) & 1023)) & 1023);
    float *recv = reinterpret_cast<float *>(sm + p.nst * stage_bytes);  // [C][RPO][cw]

    // x, the index array, A (and y with add_inputs) may come from the
    // previous kernels; a dependent expand may launch now (it reads y only
    // after its own wait, i.e. after this grid has completed).
    grid_dep_wait();
    grid_dep_launch();

    // The first stages go out before anything else: their loads do not
    // depend on the token indices.
    const uint32_t sm_base = smem_u32(sm);
#define BGMV_ISSUE_STAGE(i)                                                                 \
    do {                                                                                    \
        const int b_ = (i) % p.nst;                                                         \
        const uint32_t st_ = sm_base + (uint32_t)(b_ * stage_bytes);                        \
        mbar_arrive_expect_tx(&s_full[b_], (uint32_t)stage_bytes);                          \
        tma_load_2d(st_, &tm_x, k_begin + (i) * kBox, t0, &s_full[b_]);                     \
        tma_load_2d(st_ + kBT * 128, &tm_a, k_begin + (i) * kBox, r0, &s_full[b_]);         \
    } while (0)
    if (tid == 0) {
        for (int i = 0; i < p.nst; ++i) {
            mbar_init(&s_full[i], 1);
            mbar_init(&s_empty[i], 1);
        }
        mbar_init(&s_done, 1);
        mbar_init(&s_recv, 1);
        for (int i = 0; i < min(p.nst, nk); ++i) BGMV_ISSUE_STAGE(i);
    }
    const int t = t0 + tid;
    int my_l = -1;
    if (t < a.T) {
        const int v = a.idx ? __ldg(a.idx + t) : 0;
        if (v >= 0 && v < a.L) my_l = v;
    }
    s_l[tid] = my_l;
    __syncwarp();
    if (warp == 0) tc_alloc(&s_tmem, p.tcols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s_tmem;
    // receive barriers are initialised (fence in mbar_init) before any peer
    // stores into them: the matching wait comes before the first send
    cluster_arrive_relaxed();

    bool timed_out = false;
    if (tid == 0) {
        // TMA producer: stage i = x[t0 .. +128, k .. k+64] and the A rows;
        // stages past the ring's depth wait for the MMAs that read their buffer
        for (int i = p.nst; i < nk; ++i) {
            if (!mbar_wait_cta(&s_empty[i % p.nst], ((i / p.nst) - 1) & 1)) {
                timed_out = true;
                break;
            }
            BGMV_ISSUE_STAGE(i);
        }
    } else if (tid == 32) {
        // MMA issuer: four K = 16 steps per stage into the TMEM accumulator
        const uint32_t idesc = tc_idesc_f16(std::is_same<E, __nv_bfloat16>::value, kBT, p.n_mma);
        for (int i = 0; i < nk; ++i) {
            const int b = i % p.nst;
            if (!mbar_wait_cta(&s_full[b], (i / p.nst) & 1)) {
                timed_out = true;
                break;
            }
            tc_fence_after();
            const uint32_t xs = smem_u32(sm + b * stage_bytes), as = xs + kBT * 128;
#pragma unroll
            for (int k = 0; k < kBox / 16; ++k)
                tc_mma_f16(tmem, tc_desc_sw128(xs + 32 * k), tc_desc_sw128(as + 32 * k), idesc,
                           i > 0 || k > 0);
            tc_commit(&s_empty[b]);
        }
        tc_commit(&s_done);  // arrives once every MMA issued above is complete
    }
#undef BGMV_ISSUE_STAGE
    __syncwarp();
    if (!mbar_wait_cta(&s_done, 0)) timed_out = true;
    __syncwarp();
    tc_fence_after();

    // This lane's token: its adapter's columns of this CTA's share, 32 at a
    // time, to the CTA that finishes its row.
    const int nvalid = min(kBT, a.T - t0);
    const int li = (my_l >= l_first && my_l < l_first + l_count) ? my_l - l_first : -1;
    const int owner = tid / RPO, orow = tid - owner * RPO;
    const int nown = max(0, min(RPO, nvalid - kc * RPO));
    const uint32_t taddr = tmem + ((uint32_t)(32 * warp) << 16);
    cluster_wait();
    if (tid == 0) mbar_arrive_expect_tx(&s_recv, (uint32_t)(C * nown * cw * 4));
    const uint32_t dst = cluster_map(smem_u32(recv), (uint32_t)owner) +
                         (uint32_t)((kc * RPO + orow) * cw * 4);
    const uint32_t dst_bar = cluster_map(smem_u32(&s_recv), (uint32_t)owner);
    for (int j0 = 0; j0 < cw; j0 += 32) {  // block-uniform
        float v[32];
#pragma unroll
        for (int r = 0; r < 32; ++r) v[r] = 0.f;
        for (int q = 0; q < l_count; ++q) {  // block-uniform
            float d[32];
            tc_ld32(taddr + (uint32_t)(q * W + j0), d);
            if (q == li) {
#pragma unroll
                for (int r = 0; r < 32; ++r) v[r] = d[r];
            }
        }
        if (tid < nvalid) {
            const int nj = min(32, cw - j0);
#pragma unroll
            for (int r = 0; r < 32; r += 4)
                if (r < nj)
                    st_async_v4(dst + (uint32_t)((j0 + r) * 4),
                                make_float4(v[r], v[r + 1], v[r + 2], v[r + 3]), dst_bar);
        }
    }
    // my rows: the cluster's partials summed in rank order, then y
    if (!mbar_wait_cluster(&s_recv, 0)) timed_out = true;
    __syncwarp();
    for (int it = tid; it < nown * cw; it += kBThreads) {
        const int r = it / cw, j = it - r * cw;
        const int trow = kc * RPO + r;
        const int tl = s_l[trow];
        float sum = 0.f;
        for (int q = 0; q < C; ++q) sum += recv[(q * RPO + r) * cw + j];
        const int col = c0 + j;
        float val = 0.f;
        bool write;
        if (tl >= l_first && tl < l_first + l_count) {
            write = true;
            if (col % a.R < clamp_rank(a.ranks, tl, a.R)) val = a.scale * sum;
        } else {
            // tokens without an adapter: zeros, written by the CTAs holding adapter 0's columns
            write = tl < 0 && l_first == 0 && !a.add;
        }
        if (write) {
            float *yp = a.y + (int64_t)(t0 + trow) * a.ldy + col;
            *yp = a.add ? *yp + val : val;
        }
    }
    if (timed_out && a.status) atomicOr(a.status, LORA_PLANERR_TIMEOUT);
    // no CTA leaves while a peer may still store into its receive buffer
    __syncwarp();
    cluster_arrive();
    cluster_wait();
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tc_dealloc(tmem, p.tcols);
    }
}

// Stand-in with the shrink's block size, for the cluster-capacity queries.
__global__ void __launch_bounds__(kBThreads) bgmv_capacity_probe() {}

// ------------------------------------------------------------------ expand
// Persistent, double-buffered: every CTA walks a contiguous range of work
// items (token block x column chunk, block-major), and while item k is
// contracted and written back, the out tile and B rows of item k+1 are
// already in flight.  Y_ext is rebuilt only when the token block or the slice
// (whose y columns it holds) changes.  8 warps: warps w and w + 4 own TMEM
// lanes 32 (w % 4) .. + 31 (the block's tokens) and split the chunk's columns.
//  - out: loaded by TMA (add_inputs), updated in place in shared memory and
//    written back by TMA stores (one per 64-column box: a warp storing one
//    16-byte piece per token row would touch 32 rows per instruction);
//    rows without a LoRA term keep the values read (with add_inputs) or
//    become zeros (without); a ragged last box is stored by the threads;
//  - B_ext: cp.async pieces of 8 ranks, ranks past r_l and columns past the
//    slice zero-filled.
constexpr int kEThreads = 256;


// Shared memory: two stages of (out tile: nc / 64 boxes of 128 rows x 128 B;
// B_ext [kgroups][nc rows][128 B]), then Y_ext hi and lo [kgroups][128 rows]
// [128 B]; 128-byte swizzled K-major, 1024-byte aligned.
__host__ __device__ constexpr int expand_stage_bytes(int nc, int kgroups) {
    return nc * kBT * 2 + kgroups * nc * 128;
}
__host__ __device__ constexpr int expand_smem_bytes(int nc, int kgroups) {
    return 1024 + 2 * expand_stage_bytes(nc, kgroups) + 2 * kgroups * kBT * 128;
}

struct ExpandItem {
    int t0, s, n0, ncols;
    int64_t col0;
};

__device__ __forceinline__ ExpandItem expand_item(const BgmvExpandArgs &a, int item, int nchunks,
                                                  int nc) {
    ExpandItem it;
    const int blk = item / nchunks, chunk = item - blk * nchunks;
    int s = 0;
    while (s + 1 < a.num_slices && chunk >= a.chunk_begin[s + 1]) ++s;
    it.t0 = blk * kBT;
    it.s = s;
    it.n0 = (chunk - a.chunk_begin[s]) * nc;
    it.ncols = min(nc, a.N[s] - it.n0);  // > 0, a multiple of 8
    it.col0 = (int64_t)a.off[s] + it.n0;
    return it;
}

// One thread's part of the expand epilogue: NCOL columns (a multiple of 32)
// from column cbeg of its token row.  `so` is the row's 128-byte slice of the
// staged tile (box stride kBT * 128), `swz` the row's 16-byte swizzle.  All
// TMEM loads are issued before one wait and all staged values are read
// before the arithmetic, so the pieces are independent chains.
template <typename E, bool ADD, int NCOL>
__device__ __forceinline__ void epilogue_cols(uint32_t taddr, bool has_mma, bool live, float f,
                                              unsigned char *so, int swz, int cbeg, int ncols,
                                              int full_cols, E *orow) {
    constexpr int NP = NCOL / 8;  // 16-byte pieces
    uint32_t d[NCOL];
    if (has_mma) {
#pragma unroll
        for (int j = 0; j < NCOL / 32; ++j)
            tc_ld32_nowait(taddr + 32 * j, reinterpret_cast<uint32_t (&)[32]>(d[32 * j]));
        tc_wait_ld();
    } else {
#pragma unroll
        for (int q = 0; q < NCOL; ++q) d[q] = 0u;
    }
    if (!live) return;
    uint4 *slot[NP];
    uint4 old[NP];
#pragma unroll
    for (int g = 0; g < NP; ++g) {
        const int c = cbeg + 8 * g;
        slot[g] = reinterpret_cast<uint4 *>(so + (c >> 6) * kBT * 128 + ((((c & 63) >> 3) ^ swz) << 4));
        if (ADD) old[g] = *slot[g];
    }
#pragma unroll
    for (int g = 0; g < NP; ++g) {
        const int c = cbeg + 8 * g;
        float v[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) v[q] = f * __uint_as_float(d[8 * g + q]);
        if (ADD) {
            float o[8];
            unpack8<E>(old[g], o);
#pragma unroll
            for (int q = 0; q < 8; ++q) v[q] += o[q];
        }
        const uint4 w = pack8<E>(v);
        if (c < full_cols) *slot[g] = w;
        else if (c < ncols) st_global_v4(orow + c, w);
    }
}

// KSY: 16-wide K steps per adapter (ranks padded to RP = 16 * KSY).
template <typename E, bool ADD, int KSY>
__global__ void __launch_bounds__(kEThreads)
bgmv_expand_kernel(const __grid_constant__ CUtensorMap tm_out, const BgmvExpandArgs a, int nc,
                   int kgroups, int n_items, int nchunks) {
    constexpr int RP = 16 * KSY;
    extern __shared__ __align__(16) unsigned char smem[];
    __shared__ uint64_t s_full[2], s_mma;
    __shared__ uint32_t s_tmem;
    __shared__ int s_present;  // bit l: adapter l has a token (of nonzero rank) in the block
    __shared__ int s_l[kBT];   // adapter of each row of the block (-1: no LoRA term)
    __shared__ float s_f[kBT]; // per-row scale * 2^e of the y scaling
    const int tid = threadIdx.x, warp = tid >> 5;
    const int R = a.R;
    E *__restrict__ out = static_cast<E *>(a.out);
    const int i0 = (int)((int64_t)blockIdx.x * n_items / gridDim.x);
    const int i1 = (int)((int64_t)(blockIdx.x + 1) * n_items / gridDim.x);
    const int count = i1 - i0;
    unsigned char *sm = smem + ((1024 - (smem_u32(smem) & 1023)) & 1023);
    const int stage = expand_stage_bytes(nc, kgroups);
    unsigned char *sYh = sm + 2 * stage;
    unsigned char *sYl = sYh + kgroups * kBT * 128;
    auto sOut = [&](int b) { return sm + b * stage; };
    auto sB = [&](int b) { return sm + b * stage + nc * kBT * 2; };

    // Item j's out tile (add_inputs; rows past T zero-filled) and B rows into
    // stage b.  Thread 0 first waits until the TMA stores of the stage's
    // previous item have read it.  cp.async B pieces: one group per call and
    // thread.
    auto issue = [&](int j, int b, bool stored_before) {
        const ExpandItem it = expand_item(a, j, nchunks, nc);
        if (tid == 0) {
            if (stored_before) tma_store_wait_read();
            if (ADD) {
                const int nbox = (it.ncols + kBox - 1) / kBox;
                mbar_arrive_expect_tx(&s_full[b], (uint32_t)(nbox * kBT * 128));
                for (int i = 0; i < nbox; ++i)
                    tma_load_2d(smem_u32(sOut(b) + i * kBT * 128), &tm_out,
                                (int)(it.col0 + i * kBox), it.t0, &s_full[b]);
            }
        }
        {
            const E *Bs = static_cast<const E *>(a.B[it.s]);
            const int Ns = a.N[it.s];
            const int per_row = kgroups * 8;
            unsigned char *dstB = sB(b);
            for (int q = tid; q < nc * per_row; q += kEThreads) {
                const int n = q / per_row, c = q - n * per_row;
                const int lb = (8 * c) / RP, k = 8 * c - lb * RP;
                if (lb >= a.L) continue;
                const int nv = n < it.ncols ? min(8, clamp_rank(a.ranks, lb, R) - k) : 0;
                const E *src = nv > 0 ? Bs + ((int64_t)lb * Ns + it.n0 + n) * R + k : Bs;
                cp_async16(smem_u32(dstB + (c >> 3) * nc * 128 + n * 128 + (((c & 7) ^ (n & 7)) << 4)),
                           src, nv > 0 ? 2 * nv : 0);
            }
        }
        cp_async_commit();
    };

    if (!a.early) grid_dep_wait();  // every read after the previous kernel
    if (tid == 0) {
        mbar_init(&s_full[0], 1);
        mbar_init(&s_full[1], 1);
        mbar_init(&s_mma, 1);
        tma_prefetch_map(&tm_out);
    }
    // With early reads, the first two items' loads go out before the wait for
    // the previous kernel (the chained shrink): out and B are not written by
    // it (y is), nor is the index array (the first block's entry of this
    // thread is read now too).
    if (count > 0) issue(i0, 0, false);
    if (count > 1) issue(i0 + 1, 1, false);
    int idx_pre = -1, idx_blk = -1;
    if (count > 0) {
        idx_blk = expand_item(a, i0, nchunks, nc).t0;
        const int t = idx_blk + (tid & (kBT - 1));
        if (t < a.T) idx_pre = a.idx ? __ldg(a.idx + t) : 0;
    }
    grid_dep_wait();
    grid_dep_launch();
    // Tensor memory is taken only after that wait: a CTA holding TMEM never
    // waits on another grid.
    if (warp == 0) tc_alloc(&s_tmem, (uint32_t)nc);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s_tmem;

    const uint32_t idesc = tc_idesc_f16(std::is_same<E, __nv_bfloat16>::value, kBT, nc);
    const int r = tid & (kBT - 1), half = tid >> 7;
    int yblk = -1, yslice = -1, present = 0;
    int nmma = 0;     // phases completed on s_mma (items with MMAs)
    int waited = 0;   // items whose loads have been waited for
    bool timed_out = false;
    for (int k = 0; k < count; ++k) {
        const int b = k & 1;
        const ExpandItem it = expand_item(a, i0 + k, nchunks, nc);
        if (it.t0 != yblk || it.s != yslice) {  // block-uniform
            // Y_ext rows of the block for this slice's y columns: each token's
            // y as a hi (threads < 128) or lo (threads >= 128) part scaled by
            // 2^-e in its adapter's K block, zeros elsewhere.  The previous
            // item's MMAs are complete.
            yblk = it.t0;
            yslice = it.s;
            if (tid == 0) s_present = 0;
            const int t = it.t0 + r;
            int l = -1, rl = 0;
            if (t < a.T) {
                const int v = it.t0 == idx_blk ? idx_pre : (a.idx ? __ldg(a.idx + t) : 0);
                if (v >= 0 && v < a.L) {
                    rl = clamp_rank(a.ranks, v, R);
                    if (rl > 0) l = v;
                }
            }
            float yv[RP];
#pragma unroll
            for (int q = 0; q < RP; ++q) yv[q] = 0.f;
            float f = 0.f;
            if (l >= 0) {
                const float *yr = a.y + (int64_t)t * a.ldy + (int64_t)it.s * a.y_slice_stride;
#pragma unroll
                for (int q = 0; q < RP; q += 4)
                    if (q < rl) {
                        const float4 v = __ldcg(reinterpret_cast<const float4 *>(yr + q));
                        yv[q] = v.x;
                        yv[q + 1] = v.y;
                        yv[q + 2] = v.z;
                        yv[q + 3] = v.w;
                    }
                float m = 0.f;
#pragma unroll
                for (int q = 0; q < RP; ++q) {
                    if (q >= rl) yv[q] = 0.f;
                    m = fmaxf(m, fabsf(yv[q]));
                }
                const int e = row_exponent(m);
                f = a.scale * exp2i(e);
                const float inv = exp2i(-e);
#pragma unroll
                for (int q = 0; q < RP; ++q) yv[q] *= inv;
            }
            __syncthreads();  // s_present reset; nobody reads the previous rows now
            if (half == 0) {
                s_l[r] = l;
                s_f[r] = f;
                if (l >= 0) atomicOr(&s_present, 1 << l);
            }
            unsigned char *dstY = half ? sYl : sYh;
            const int cl0 = l >= 0 ? l * (RP / 8) : -RP;  // first 16-byte piece of the block
            for (int c = 0; c < kgroups * 8; ++c) {
                if (c >= cl0 && c < cl0 + RP / 8) continue;
                *reinterpret_cast<uint4 *>(dstY + (c >> 3) * kBT * 128 + r * 128 +
                                           (((c & 7) ^ (r & 7)) << 4)) = make_uint4(0, 0, 0, 0);
            }
            if (l >= 0) {
#pragma unroll
                for (int j = 0; j < RP / 8; ++j) {
                    float v[8];
#pragma unroll
                    for (int q = 0; q < 8; ++q) v[q] = yv[8 * j + q];
                    uint4 hi, lo;
                    split_hilo8<E>(v, hi, lo);
                    const int c = cl0 + j;
                    *reinterpret_cast<uint4 *>(dstY + (c >> 3) * kBT * 128 + r * 128 +
                                               (((c & 7) ^ (r & 7)) << 4)) = half ? lo : hi;
                }
            }
        }
        // this item's B pieces (cp.async; one newer group may be in flight)
        if (k + 1 < count) cp_async_wait<1>();
        else cp_async_wait<0>();
        fence_proxy_async_smem();  // Y (plain stores) and B (cp.async) -> tensor-core reads
        __syncthreads();
        present = s_present;
        bool to = false;
        if (ADD && !mbar_wait_cta(&s_full[b], (k >> 1) & 1)) to = true;
        if (!to) waited = k + 1;
        if (tid == 0 && present) {
            tc_fence_after();
            bool acc = false;
            for (int lb = 0; lb < a.L; ++lb) {
                if (!((present >> lb) & 1)) continue;
#pragma unroll
                for (int ks = 0; ks < KSY; ++ks) {
                    const int kpos = lb * RP + 16 * ks;
                    const uint32_t g = (uint32_t)(kpos >> 6), kb = (uint32_t)((kpos & 63) * 2);
                    const uint32_t yh = smem_u32(sYh) + g * kBT * 128 + kb;
                    const uint32_t yl = smem_u32(sYl) + g * kBT * 128 + kb;
                    const uint32_t bb = smem_u32(sB(b)) + g * (uint32_t)nc * 128 + kb;
                    tc_mma_f16(tmem, tc_desc_sw128(yh), tc_desc_sw128(bb), idesc, acc);
                    tc_mma_f16(tmem, tc_desc_sw128(yl), tc_desc_sw128(bb), idesc, true);
                    acc = true;
                }
            }
            tc_commit(&s_mma);
        }
        // the MMA barrier completes one phase per item that has MMAs
        if (present) {
            if (!mbar_wait_cta(&s_mma, (uint32_t)(nmma & 1))) to = true;
            ++nmma;
        }
        if (__syncthreads_or(to)) {  // never expected: flag it and leave out untouched
            if (tid == 0 && a.status) atomicOr(a.status, LORA_PLANERR_TIMEOUT);
            timed_out = true;
            break;
        }
        tc_fence_after();
        // epilogue: this thread's token row, its half of the chunk's columns
        // (32 or 64), all TMEM loads and staged values in flight at once;
        // full 64-column boxes are updated in shared memory for the TMA
        // stores, the columns of a ragged last box are stored directly
        const int full_cols = (it.ncols / kBox) * kBox;
        {
            const int t = it.t0 + r, l = s_l[r];
            const bool live = t < a.T && (l >= 0 || !ADD);
            const float f = s_f[r];
            const int cbeg = half * (nc / 2);
            const uint32_t taddr = tmem + ((uint32_t)(32 * (warp & 3)) << 16) + (uint32_t)cbeg;
            unsigned char *so = sOut(b) + r * 128;
            const int swz = r & 7;
            if (nc == 128) {
                if (cbeg < it.ncols)
                    epilogue_cols<E, ADD, 64>(taddr, present != 0, live, f, so, swz, cbeg,
                                              it.ncols, full_cols, out + (int64_t)t * a.ldo + it.col0);
            } else if (cbeg < it.ncols) {
                epilogue_cols<E, ADD, 32>(taddr, present != 0, live, f, so, swz, cbeg, it.ncols,
                                          full_cols, out + (int64_t)t * a.ldo + it.col0);
            }
        }
        fence_proxy_async_smem();  // the updated tile -> the TMA stores
        tc_fence_before();
        __syncthreads();  // stage b's B, TMEM and the block's rows are free again
        if (tid == 0 && full_cols > 0) {
            for (int i = 0; i < full_cols / kBox; ++i)
                tma_store_2d(&tm_out, (int)(it.col0 + i * kBox), it.t0,
                             smem_u32(sOut(b) + i * kBT * 128));
            tma_store_commit();
        }
        if (k + 2 < count) issue(i0 + k + 2, b, full_cols > 0);
    }
    // no copy into or out of this CTA's shared memory may be in flight when it
    // exits (after a timed-out wait: one more bounded wait per load not yet seen)
    cp_async_wait<0>();
    if (ADD && timed_out) {
        const int issued = min(count, waited + 2);
        for (int k = waited; k < issued; ++k) mbar_wait_cta(&s_full[k & 1], (k >> 1) & 1);
    }
    if (timed_out && nmma > 0) mbar_wait_cta(&s_mma, (uint32_t)((nmma - 1) & 1));
    if (tid == 0) tma_store_wait_all();
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tc_dealloc(tmem, (uint32_t)nc);
    }
}

// ------------------------------------------------------------------ expand, small ranks
// One 64-token x 128-column tile per CTA (fma_expand.cuh): with early reads
// everything that does not depend on y is staged before the wait for the
// previous kernel.
template <typename E, bool ADD, int RK8>
__global__ void __launch_bounds__(kFThreads)
bgmv_expand_fma_kernel(const BgmvExpandArgs a, int nchunks) {
    extern __shared__ __align__(16) unsigned char smem[];
    __shared__ int s_l[kFRows];
    __shared__ __align__(16) float s_y[kFRows][8 * RK8];
    const FmaTile tt = fma_tile(a, (int)blockIdx.x, nchunks);
    uint4 *sB = reinterpret_cast<uint4 *>(smem);  // [adapters][RK8][kFCols]
    uint32_t old[8][2];
    if (!a.early) grid_dep_wait();  // every read after the previous kernel
    fma_stage<E, ADD, RK8>(a, tt, sB, s_l, old);
    // y rows come from the previous kernel (the shrink)
    grid_dep_wait();
    grid_dep_launch();
    fma_stage_y<RK8>(a, tt, s_y);
    cp_async_commit();
    cp_async_wait<0>();
    __syncthreads();
    fma_finish<E, ADD, RK8>(a, tt, sB, s_y, s_l, old);
}

// ------------------------------------------------------------------ expand, one adapter
// No token index: every token uses adapter 0, so there is nothing to mask or
// look up (the mask-free single-adapter case).  Each thread keeps the B rows
// of its two output columns in registers as fp32 and streams the tile's
// token rows past them: per row one broadcast read of y from shared memory
// and 2r multiply-adds, no shared-memory traffic for B.  A CTA covers 64
// tokens x 64 columns of one slice (lane j: columns 2j, 2j+1; warp w: rows
// w, w + 8, ...), stored as coalesced 4-byte pairs.
constexpr int kDRows = 64, kDCols = 64;

template <typename E, bool ADD, int RK8>
__global__ void __launch_bounds__(kFThreads)
bgmv_expand_dense_kernel(const BgmvExpandArgs a, int nchunks) {
    constexpr int RK = 8 * RK8;  // == R (a multiple of 8)
    __shared__ __align__(16) float s_y[kDRows][RK];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int chunk = (int)(blockIdx.x % (unsigned)nchunks);
    const int t0 = (int)(blockIdx.x / (unsigned)nchunks) * kDRows;
    int s = 0;
    while (s + 1 < a.num_slices && chunk >= a.chunk_begin[s + 1]) ++s;
    const int n0 = (chunk - a.chunk_begin[s]) * kDCols;
    const int c = n0 + 2 * lane;  // this thread's first column within the slice
    const bool ok = c < a.N[s];    // (slice widths are even)
    if (!a.early) grid_dep_wait();  // every read after the previous kernel
    const int rl = clamp_rank(a.ranks, 0, a.R);
    const int64_t col = (int64_t)a.off[s] + c;
    // B rows of columns c, c + 1 (ranks past r_0 as zeros)
    float b0[RK], b1[RK];
    {
        const E *Bs = static_cast<const E *>(a.B[s]);
#pragma unroll
        for (int k8 = 0; k8 < RK8; ++k8) {
            uint4 p0 = make_uint4(0u, 0u, 0u, 0u), p1 = p0;
            if (ok && 8 * k8 < rl) {
                p0 = __ldg(reinterpret_cast<const uint4 *>(Bs + (int64_t)c * a.R + 8 * k8));
                p1 = __ldg(reinterpret_cast<const uint4 *>(Bs + (int64_t)(c + 1) * a.R + 8 * k8));
            }
            float v0[8], v1[8];
            unpack8<E>(p0, v0);
            unpack8<E>(p1, v1);
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                b0[8 * k8 + e] = 8 * k8 + e < rl ? v0[e] : 0.f;
                b1[8 * k8 + e] = 8 * k8 + e < rl ? v1[e] : 0.f;
            }
        }
    }
    E *__restrict__ out = static_cast<E *>(a.out);
    uint32_t old[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        old[i] = 0u;
        const int t = t0 + i * 8 + warp;
        if (ADD && ok && t < a.T)
            old[i] = __ldcs(reinterpret_cast<const uint32_t *>(out + (int64_t)t * a.ldo + col));
    }
    // y rows come from the previous kernel (the shrink)
    grid_dep_wait();
    grid_dep_launch();
    // each warp stages the y rows it computes (rows warp, warp + 8, ...): no
    // block-wide barrier
    for (int q = lane; q < (kDRows / 8) * (RK / 4); q += 32) {
        const int i = q / (RK / 4), k4 = q - i * (RK / 4);
        const int rr = i * 8 + warp, t = t0 + rr;
        const bool in = t < a.T && 4 * k4 < rl;  // ranks past r_0 read as zeros
        const float *src =
            in ? a.y + (int64_t)t * a.ldy + (int64_t)s * a.y_slice_stride + 4 * k4 : a.y;
        cp_async16(smem_u32(&s_y[rr][4 * k4]), src, in ? 4 * min(4, rl - 4 * k4) : 0);
    }
    cp_async_commit();
    cp_async_wait<0>();
    __syncwarp();
    if (!ok || (ADD && rl == 0)) return;  // (rank 0 with add_inputs: out stays as it is)
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int rr = i * 8 + warp, t = t0 + rr;
        if (t < a.T) {
            float acc0 = 0.f, acc1 = 0.f;
#pragma unroll
            for (int k4 = 0; k4 < RK / 4; ++k4) {
                const float4 yv = *reinterpret_cast<const float4 *>(&s_y[rr][4 * k4]);
                acc0 = fmaf(yv.x, b0[4 * k4], acc0);
                acc0 = fmaf(yv.y, b0[4 * k4 + 1], acc0);
                acc0 = fmaf(yv.z, b0[4 * k4 + 2], acc0);
                acc0 = fmaf(yv.w, b0[4 * k4 + 3], acc0);
                acc1 = fmaf(yv.x, b1[4 * k4], acc1);
                acc1 = fmaf(yv.y, b1[4 * k4 + 1], acc1);
                acc1 = fmaf(yv.z, b1[4 * k4 + 2], acc1);
                acc1 = fmaf(yv.w, b1[4 * k4 + 3], acc1);
            }
            float v0 = a.scale * acc0, v1 = a.scale * acc1;
            if (ADD) {
                const float2 o = Pack<E>::unpack(old[i]);
                v0 += o.x;
                v1 += o.y;
            }
            *reinterpret_cast<uint32_t *>(out + (int64_t)t * a.ldo + col) = Pack<E>::pack(v0, v1);
        }
    }
}

using DenseFn = void (*)(const BgmvExpandArgs, int);
template <typename E, bool ADD>
DenseFn dense_fn(int rk8) {
    switch (rk8) {
        case 1: return bgmv_expand_dense_kernel<E, ADD, 1>;
        case 2: return bgmv_expand_dense_kernel<E, ADD, 2>;
        case 3: return bgmv_expand_dense_kernel<E, ADD, 3>;
        default: return bgmv_expand_dense_kernel<E, ADD, 4>;
    }
}
DenseFn dense_fn(int dt, bool add, int rk8) {
    if (dt == LORA_F16) return add ? dense_fn<__half, true>(rk8) : dense_fn<__half, false>(rk8);
    return add ? dense_fn<__nv_bfloat16, true>(rk8) : dense_fn<__nv_bfloat16, false>(rk8);
}

using FmaFn = void (*)(const BgmvExpandArgs, int);
template <typename E, bool ADD>
FmaFn fma_fn(int rk8) {
    switch (rk8) {
        case 1: return bgmv_expand_fma_kernel<E, ADD, 1>;
        case 2: return bgmv_expand_fma_kernel<E, ADD, 2>;
        case 3: return bgmv_expand_fma_kernel<E, ADD, 3>;
        default: return bgmv_expand_fma_kernel<E, ADD, 4>;
    }
}
FmaFn fma_fn(int dt, bool add, int rk8) {
    if (dt == LORA_F16) return add ? fma_fn<__half, true>(rk8) : fma_fn<__half, false>(rk8);
    return add ? fma_fn<__nv_bfloat16, true>(rk8) : fma_fn<__nv_bfloat16, false>(rk8);
}
// Dispatch: the FMA kernel for ranks up to 32 and batches up to 256 tokens.
// Measured on the Llama-3-8B q/k/v decode shapes (rank 16, 4 adapters),
// chained after the shrink: 10.4 / 11.8 / 13.9 us at 16 / 128 / 256 tokens
// against 11.3 / 12.1 / 15.8 us with the tensor-core expand; from 512
// tokens on its shared-memory reads of B (2r bytes per output element) cost
// more than the tensor-core path (21.4 against 19.0 us).
constexpr int kFmaMaxRank = 32;
constexpr int kFmaMaxTokens = 256;

using ExpandFn = void (*)(const CUtensorMap, const BgmvExpandArgs, int, int, int, int);
template <typename E, bool ADD>
ExpandFn expand_fn(int ksy) {
    switch (ksy) {
        case 1: return bgmv_expand_kernel<E, ADD, 1>;
        case 2: return bgmv_expand_kernel<E, ADD, 2>;
        case 3: return bgmv_expand_kernel<E, ADD, 3>;
        default: return bgmv_expand_kernel<E, ADD, 4>;
    }
}
ExpandFn expand_fn(int dt, bool add, int ksy) {
    if (dt == LORA_F16) return add ? expand_fn<__half, true>(ksy) : expand_fn<__half, false>(ksy);
    return add ? expand_fn<__nv_bfloat16, true>(ksy) : expand_fn<__nv_bfloat16, false>(ksy);
}

using ShrinkFn = void (*)(const CUtensorMap, const CUtensorMap, const BgmvShrinkArgs, const ShrinkSplit);
ShrinkFn shrink_fn(int dt) {
    return dt == LORA_F16 ? bgmv_shrink_kernel<__half> : bgmv_shrink_kernel<__nv_bfloat16>;
}

// Cluster capacity: CTAs of clusters of 1, 2, 4, 8, 16 resident at once,
// [two per SM (<= kShrinkSmemCap of shared memory) or one][log2 cluster].
int g_cluster_ctas[2][5] = {};
int g_sm_count = 0;
int g_smem_sm = 0, g_smem_reserved = 0, g_shrink_static = 0;

// Dynamic shared memory of a shrink CTA, raised where needed so that the
// CTAs one SM holds never ask for more than its 512 TMEM columns together: a
// CTA waiting in tcgen05.alloc could otherwise hold up a cluster peer that
// itself holds columns.
int shrink_smem_for_tmem(int dyn, int tcols) {
    const int max_ctas = 512 / tcols;
    const int per_cta = g_smem_sm / (max_ctas + 1) + 1;  // more than this fits max_ctas at most
    return std::max(dyn, per_cta - g_shrink_static - g_smem_reserved);
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

}  // namespace

cudaError_t configure_bgmv_kernels(const DeviceInfo &dev) {
    g_sm_count = dev.sm_count;
    int devid = 0;
    cudaError_t e = cudaGetDevice(&devid);
    if (e == cudaSuccess)
        e = cudaDeviceGetAttribute(&g_smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, devid);
    if (e == cudaSuccess)
        e = cudaDeviceGetAttribute(&g_smem_reserved, cudaDevAttrReservedSharedMemoryPerBlock, devid);
    int optin = 0;
    if (e == cudaSuccess)
        e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, devid);
    if (e == cudaSuccess) {
        cudaFuncAttributes fa;
        e = cudaFuncGetAttributes(&fa, shrink_fn(LORA_BF16));
        g_shrink_static = (int)fa.sharedSizeBytes;
    }
    // dynamic shared memory allowed per block: the opt-in limit less static use
    const int big = optin - g_shrink_static;
    for (int dt = 0; dt < 2 && e == cudaSuccess; ++dt) {
        e = cudaFuncSetAttribute(shrink_fn(dt), cudaFuncAttributeMaxDynamicSharedMemorySize, big);
        if (e == cudaSuccess && dev.max_cluster > 8)
            e = cudaFuncSetAttribute(shrink_fn(dt), cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        for (int add = 0; add < 2 && e == cudaSuccess; ++add)
            for (int ksy = 1; ksy <= 4 && e == cudaSuccess; ++ksy)
                e = cudaFuncSetAttribute(expand_fn(dt, add != 0, ksy),
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         expand_smem_bytes(128, 2));
    }
    for (int dt = 0; dt < 2 && e == cudaSuccess; ++dt)
        for (int add = 0; add < 2 && e == cudaSuccess; ++add)
            for (int rk8 = 1; rk8 <= 4 && e == cudaSuccess; ++rk8)
                e = cudaFuncSetAttribute(fma_fn(dt, add != 0, rk8),
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         fma_b_bytes(LORA_BGMV_MAX_ADAPTERS, 4));
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(bgmv_capacity_probe, cudaFuncAttributeMaxDynamicSharedMemorySize, optin);
    if (e == cudaSuccess && dev.max_cluster > 8)
        e = cudaFuncSetAttribute(bgmv_capacity_probe, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    for (int two = 0; two < 2 && e == cudaSuccess; ++two) {
        for (int lc = 0; lc < 5 && e == cudaSuccess; ++lc) {
            const int C = 1 << lc;
            if (C > dev.max_cluster) break;
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3(C, 1, 1);
            cfg.blockDim = dim3(kBThreads);
            cfg.dynamicSmemBytes = two ? kShrinkSmemCap - 8 * 1024 : big - 8 * 1024;
            cudaLaunchAttribute attr[1];
            attr[0].id = cudaLaunchAttributeClusterDimension;
            attr[0].val.clusterDim.x = C;
            attr[0].val.clusterDim.y = 1;
            attr[0].val.clusterDim.z = 1;
            cfg.attrs = attr;
            cfg.numAttrs = 1;
            int n = 0;
            e = cudaOccupancyMaxActiveClusters(&n, bgmv_capacity_probe, &cfg);
            g_cluster_ctas[two][lc] = n * C;
        }
    }
    return e;
}

const char *bgmv_shrink_supported(const BgmvShrinkArgs &a) {
    const int W = a.S * a.R;
    if (!aligned16(a.x) || a.ldx % 8 != 0) return "x must be 16-byte aligned with ldx a multiple of 8";
    if (!aligned16(a.A) || a.H % 8 != 0) return "A must be 16-byte aligned with H a multiple of 8";
    if (W % 8 != 0) return "num_slices * R must be a multiple of 8";
    return nullptr;
}

const char *bgmv_expand_supported(const BgmvExpandArgs &a) {
    const int RP = (a.R + 15) / 16 * 16;
    if (a.R % 8 != 0) return "R must be a multiple of 8";
    if (RP > 64) return "R above 64 (use the grouped operators)";
    if (a.L * RP > 128) return "L * R (ranks padded to 16) above 128 (use the grouped operators)";
    if (!aligned16(a.y) || a.ldy % 4 != 0 || a.y_slice_stride % 4 != 0)
        return "y must be 16-byte aligned with ldy and y_slice_stride multiples of 4";
    if (!aligned16(a.out) || a.ldo % 8 != 0) return "out must be 16-byte aligned with ldo a multiple of 8";
    for (int s = 0; s < a.num_slices; ++s)
        if (a.N[s] > 0 && (a.N[s] % 8 != 0 || a.off[s] % 8 != 0 || !aligned16(a.B[s])))
            return "slice widths and offsets must be multiples of 8, B_s 16-byte aligned";
    return nullptr;
}

cudaError_t launch_bgmv_shrink(lora_dtype_t dt, const BgmvShrinkArgs &a, const DeviceInfo &dev,
                               cudaStream_t stream, bool pdl) {
    if (a.T == 0) return cudaSuccess;
    const int W = a.S * a.R;
    const int blocks = (a.T + kBT - 1) / kBT;
    // K split over a cluster: the largest power of two leaving >= 128 K per CTA
    int C = 1;
    while (2 * C <= dev.max_cluster && a.H / (2 * C) >= 2 * kBox) C *= 2;
    int kc_len = ((a.H + C - 1) / C + kBox - 1) / kBox * kBox;
    while (C > 1 && (long long)(C - 1) * kc_len >= a.H) {  // every CTA gets some K
        C /= 2;
        kc_len = ((a.H + C - 1) / C + kBox - 1) / kBox * kBox;
    }
    int lc = 0;
    while ((1 << lc) < C) ++lc;
    // Shares of the y columns, coarse to fine: whole adapters (zk of them,
    // N = zk * W <= 256), then column ranges of one adapter.  Measured on the
    // decode q/k/v batches (T = 16 .. 1024), the coarsest share is the best or
    // within 2 %: finer shares re-read x from L2 and, for large batches,
    // overflow the wave of clusters the GPU holds.
    struct Cand {
        int zk, zc, cw, Z;
    } cands[24];
    int nc = 0;
    if (W <= kMaxCw) {
        for (int zk = a.L; zk >= 1; zk = zk > 1 ? (zk + 1) / 2 : 0) {
            if ((zk > 1 && W % 16 != 0) || (zk * W + 15) / 16 * 16 > 256 ||
                (zk - 1) * W + (W + 31) / 32 * 32 > 256) {
                if (zk == 1) break;
                continue;
            }
            cands[nc++] = {zk, 1, W, (a.L + zk - 1) / zk};
            if (zk == 1) break;
        }
    }
    for (int cw = kMaxCw; cw >= 16 && nc < 24; cw /= 2)
        if (cw < W) cands[nc++] = {1, (W + cw - 1) / cw, cw, a.L * ((W + cw - 1) / cw)};
    if (nc == 0) return cudaErrorInvalidValue;  // unreachable: W % 8 == 0 gives a column share
    const int pick = 0;
    if (cands[pick].Z > 65535) return cudaErrorInvalidConfiguration;
    ShrinkSplit p{};
    p.kc_len = kc_len;
    p.zk = cands[pick].zk;
    p.zc = cands[pick].zc;
    p.cw = cands[pick].cw;
    p.n_mma = ((p.zk - 1) * W + p.cw + 15) / 16 * 16;
    const int tneed = (p.zk - 1) * W + (p.cw + 31) / 32 * 32;
    p.tcols = 32;
    while ((int)p.tcols < tneed) p.tcols *= 2;
    // Stage ring: the deepest (up to the CTA's whole K range, at most 4
    // stages in flight) whose shared memory still lets the whole grid of
    // clusters be resident at once (one CTA per SM above kShrinkSmemCap)
    const int nk = (kc_len + kBox - 1) / kBox;
    const int stage = kBT * 128 + p.n_mma * 128, recv = kBT * p.cw * 4;
    const long long ctas = (long long)blocks * C * cands[pick].Z;
    int smem = 0;
    for (p.nst = std::min(kMaxStages, nk); ; --p.nst) {
        smem = shrink_smem_for_tmem(1024 + p.nst * stage + recv, p.tcols);
        const int cap = g_cluster_ctas[smem <= kShrinkSmemCap ? 1 : 0][lc];
        if (ctas <= cap || p.nst <= std::min(2, nk)) break;
    }

    CUtensorMap tx, ta;
    cudaError_t e = make_map(&tx, dt, a.x, (uint64_t)a.T, (uint64_t)a.H, (uint64_t)a.ldx, kBT);
    if (e == cudaSuccess)
        e = make_map(&ta, dt, a.A, (uint64_t)a.L * W, (uint64_t)a.H, (uint64_t)a.H, (uint32_t)p.n_mma);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(C, blocks, cands[pick].Z);
    cfg.blockDim = dim3(kBThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = C;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 2 : 1;
    return cudaLaunchKernelEx(&cfg, shrink_fn(dt), tx, ta, a, p);
}

cudaError_t launch_bgmv_expand(lora_dtype_t dt, const BgmvExpandArgs &a_in, const DeviceInfo &dev,
                               cudaStream_t stream, bool pdl) {
    BgmvExpandArgs a = a_in;
    if (a.T == 0) return cudaSuccess;
    if (a.idx == nullptr && a.R <= kFmaMaxRank) {
        // one adapter: B in registers, 64 tokens x 64 columns per CTA
        a.chunk_begin[0] = 0;
        for (int s = 0; s < a.num_slices; ++s)
            a.chunk_begin[s + 1] = a.chunk_begin[s] + (a.N[s] + kDCols - 1) / kDCols;
        for (int s = a.num_slices; s < LORA_MAX_SLICES; ++s) a.chunk_begin[s + 1] = a.chunk_begin[s];
        const int nchunks = a.chunk_begin[a.num_slices];
        if (nchunks == 0) return cudaSuccess;
        const long long rblocks = (a.T + kDRows - 1) / kDRows;
        if (rblocks * nchunks > INT_MAX) return cudaErrorInvalidConfiguration;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)(rblocks * nchunks));
        cfg.blockDim = dim3(kFThreads);
        cfg.stream = stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = pdl ? 1 : 0;
        return cudaLaunchKernelEx(&cfg, dense_fn(dt, a.add != 0, (a.R + 7) / 8), a, nchunks);
    }
    if (a.R <= kFmaMaxRank && a.T <= kFmaMaxTokens) {
        // fp32 FMA kernel: 64 tokens x 128 columns per CTA
        const int nchunks = fma_set_chunks(a);
        if (nchunks == 0) return cudaSuccess;
        const long long rblocks = (a.T + kFRows - 1) / kFRows;
        if (rblocks * nchunks > INT_MAX) return cudaErrorInvalidConfiguration;
        const int rk8 = (a.R + 7) / 8;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)(rblocks * nchunks));
        cfg.blockDim = dim3(kFThreads);
        cfg.dynamicSmemBytes = (size_t)fma_b_bytes(a.idx ? a.L : 1, rk8);
        cfg.stream = stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = pdl ? 1 : 0;
        return cudaLaunchKernelEx(&cfg, fma_fn(dt, a.add != 0, rk8), a, nchunks);
    }
    const int RP = (a.R + 15) / 16 * 16;
    const int kgroups = (a.L * RP + 63) / 64;
    const long long blocks = (a.T + kBT - 1) / kBT;
    auto chunks = [&](int nc) {
        long long n = 0;
        for (int s = 0; s < a.num_slices; ++s) n += (a.N[s] + nc - 1) / nc;
        return n;
    };
    // 128 output columns per work item; 64 when there are fewer 128-column
    // items than SMs (more, smaller items spread a small batch wider)
    int nc = 128;
    if (blocks * chunks(128) < dev.sm_count) nc = 64;
    a.chunk_begin[0] = 0;
    for (int s = 0; s < a.num_slices; ++s) a.chunk_begin[s + 1] = a.chunk_begin[s] + (a.N[s] + nc - 1) / nc;
    for (int s = a.num_slices; s < LORA_MAX_SLICES; ++s) a.chunk_begin[s + 1] = a.chunk_begin[s];
    const int nchunks = a.chunk_begin[a.num_slices];
    if (nchunks == 0) return cudaSuccess;
    const long long items = blocks * nchunks;
    if (items > INT_MAX) return cudaErrorInvalidConfiguration;
    const int smem = expand_smem_bytes(nc, kgroups);
    // persistent: as many CTAs as the GPU holds at once, at most one per item
    const int per_sm = std::max(1, std::min(2, (g_smem_sm - 2048) / (smem + g_smem_reserved)));
    const int grid = (int)std::min<long long>(items, (long long)per_sm * dev.sm_count);
    CUtensorMap tm_out;
    int used = 0;
    for (int s = 0; s < a.num_slices; ++s)
        if (a.N[s] > 0) used = std::max(used, a.off[s] + a.N[s]);
    cudaError_t e = make_map(&tm_out, dt, a.out, (uint64_t)a.T, (uint64_t)used, (uint64_t)a.ldo, kBT);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kEThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, expand_fn(dt, a.add != 0, RP / 16), tm_out, a, nc, kgroups,
                              (int)items, nchunks);
}

}  // namespace lora
