// One-launch decode pair: shrink -> expand_slice for batches of at most 256
// tokens in a single cooperative launch.
//
// Splitting the LoRA computation into a shrink launch and an expand launch
// (vLLM PR #15655, the summary list) costs, on every layer, a second launch
// and a hand-off between grids; at decode sizes those fixed costs are most of
// the time.  Here one grid (clusters of 8 CTAs, at most one CTA per SM) runs
// its phases separated by the grid-wide barrier of a cooperative launch (the
// launch makes every CTA resident at once, so the barrier completes, and no
// CTA leaves before it):
//
//   0. each CTA reads the token indices, requests what needs none (its shrink
//      unit's A rows, its first expand tile's old out values), groups the
//      batch's tokens by adapter in token order (one token per thread),
//      zeroes the y rows of tokens without a LoRA term and requests the x
//      rows of its unit's first token group;
//   1. shrink units (adapter l, slice s), one per cluster of 8 CTAs that
//      split K: each CTA's partial products x[tokens, K range] .
//      A[l][sR:(s+1)R, K range]^T come from mma.sync m16n8k16 (fp32
//      accumulate) and go to the CTA that owns the row in shared memory
//      (distributed shared memory, 8 rows per CTA); after a cluster barrier
//      the owner adds the 8 partials in CTA order and writes y;
//   -- grid barrier: y is complete --
//   2. expand tiles, as in the plan-free FMA expand (fma_expand.cuh).
//
// The result is the one of lora_bgmv_shrink + lora_bgmv_expand_slice (the
// shrink of the "Punica: Multi-Tenant LoRA Serving" BGMV operator and the
// expand of vLLM PR #11579's expand_slice); y's partial sums are added in a
// fixed order, so the result does not change from run to run.
#include <cooperative_groups.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>

#include "common.cuh"
#include "fma_expand.cuh"
#include "frag.cuh"
#include "kernels.h"

namespace lora {
namespace {

namespace cg = cooperative_groups;

constexpr int kSK = 64;            // K columns per shrink stage (128-byte rows)
constexpr int kCK = 8;             // CTAs of a cluster, splitting K
constexpr int kPassStages = 8;     // stages held in shared memory at once
constexpr int kSRows = 64;         // tokens per shrink group (4 m-tiles)
constexpr int kFusedMaxT = kFThreads;  // the grouping takes one token per thread
constexpr int kFusedMaxRank = 32;      // the FMA expand tile

// 16-byte chunk c of row r in a [rows][64] 16-bit stage (128-byte rows): the
// chunk index XOR-ed with the row, so eight rows read by one ldmatrix phase
// fall in eight different bank groups.
__device__ __forceinline__ uint32_t stage_off(int r, int c) { return r * 128 + ((c ^ (r & 7)) << 4); }

// Shared memory of phase 1 (A and x stages of one pass) and of phase 2 (the
// B tile) is the same region.
__host__ __device__ constexpr int fused_smem_bytes(int nl, int rk8) {
    return fma_b_bytes(nl, rk8) > kPassStages * (kSRows + 8 * rk8) * 128
               ? fma_b_bytes(nl, rk8)
               : kPassStages * (kSRows + 8 * rk8) * 128;
}

// cp.async of stages [st0, st1) of the CTA's K range: A[l][s*R + j, :] for
// j < R (rows past r_l read as zeros) and, when `with_x`, x rows of up to 64
// tokens (s_tok[tok0 ..], or tokens tok0 .. when s_tok is null; rows past
// cnt read as zeros).  Left uncommitted.
template <typename E>
__device__ __forceinline__ void issue_pass(const BgmvShrinkArgs &a, int l, int s, int kb, int k1,
                                           int st0, int st1, bool with_a, bool with_x,
                                           const int *s_tok, int tok0, int cnt,
                                           unsigned char *sX, unsigned char *sA) {
    const int R = a.R, W = a.S * a.R;
    const int ns = st1 - st0;
    // Only rows that feed a kept result are copied: A rows j < r_l and x rows
    // r < cnt (the other rows of a 16-row m-tile or an n-tile give products
    // that are never read).  Columns past H are zero-filled, since they meet
    // valid rows in the contraction.
    if (with_a) {
        const E *A = static_cast<const E *>(a.A);
        const int rl = clamp_rank(a.ranks, l, R);
        const uint32_t ab = smem_u32(sA);
        for (int q = threadIdx.x; q < ns * rl * 8; q += kFThreads) {
            const int st = q / (rl * 8), rem = q - st * rl * 8, j = rem >> 3, c = rem & 7;
            const int k = kb + (st0 + st) * kSK + 8 * c;
            const bool ok = k < k1;
            const E *src = ok ? A + ((int64_t)l * W + s * R + j) * a.H + k : A;
            cp_async16(ab + st * R * 128 + stage_off(j, c), src, ok ? 16 : 0);
        }
    }
    if (with_x) {
        const E *x = static_cast<const E *>(a.x);
        const uint32_t xb = smem_u32(sX);
        for (int q = threadIdx.x; q < ns * cnt * 8; q += kFThreads) {
            const int st = q / (cnt * 8), rem = q - st * cnt * 8, r = rem >> 3, c = rem & 7;
            const int k = kb + (st0 + st) * kSK + 8 * c;
            const bool ok = k < k1;
            const int t = s_tok ? s_tok[tok0 + r] : tok0 + r;
            const E *src = ok ? x + (int64_t)t * a.ldx + k : x;
            cp_async16(xb + st * kSRows * 128 + stage_off(r, c), src, ok ? 16 : 0);
        }
    }
}

__device__ __forceinline__ void st_cluster_v4(uint32_t addr, float4 v) {
    asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};\n" ::"r"(addr), "f"(v.x),
                 "f"(v.y), "f"(v.z), "f"(v.w)
                 : "memory");
}

template <typename E, bool ADD, int RK8>
__global__ void __launch_bounds__(kFThreads, 1)
bgmv_fused_kernel(const BgmvShrinkArgs sa, const BgmvExpandArgs ea, int nchunks, int n_items) {
    constexpr int RK = 8 * RK8;  // == R (a multiple of 8)
    extern __shared__ __align__(16) unsigned char smem[];
    __shared__ __align__(16) float s_y[kFRows][RK];
    __shared__ __align__(16) float s_recv[kCK][kSRows / kCK][RK];  // partial rows from each CTA
    __shared__ __align__(16) float s_part[2 * kSRows][RK];        // warps' partials (K split)
    __shared__ int s_l[kFRows];
    __shared__ int s_map[kFusedMaxT];  // adapter of each token, -1 = none
    __shared__ int s_tok[kFusedMaxT];  // tokens grouped by adapter, in token order
    __shared__ int s_wc[LORA_BGMV_MAX_ADAPTERS][kFThreads / 32];
    __shared__ int s_cnt[LORA_BGMV_MAX_ADAPTERS], s_beg[LORA_BGMV_MAX_ADAPTERS];
    cg::grid_group grid = cg::this_grid();
    // Launched without the cooperative attribute (not by this library), the
    // grid barrier has no storage: write nothing rather than wait on it.
    if (!grid.is_valid()) return;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int T = sa.T, L = sa.L, R = sa.R, H = sa.H, S = sa.S, W = sa.S * sa.R;
    const int cr = (int)cluster_rank();              // this CTA's K range
    const int q0 = (int)blockIdx.x / kCK;            // this cluster
    const int nclusters = (int)gridDim.x / kCK;
    const int n_units = L * S;                       // (adapter, slice)
    const int kc_len = ((H + kCK - 1) / kCK + kSK - 1) / kSK * kSK;
    const int kb = min(H, cr * kc_len), k1 = min(H, kb + kc_len);
    const int nst = (k1 - kb + kSK - 1) / kSK;       // may be 0 for small H
    const int npass = (nst + kPassStages - 1) / kPassStages;
    // Up to 64 tokens, every unit takes all of them (rows of other adapters
    // are computed and dropped), so x needs no token index; above, a unit
    // takes its adapter's tokens, gathered, in groups of 64.
    const bool dense = T <= kSRows;
    uint4 *sB = reinterpret_cast<uint4 *>(smem);    // phase 2
    unsigned char *sX = smem;                        // phase 1: [kPassStages][64][128 B]
    unsigned char *sA = smem + kPassStages * kSRows * 128;  // [kPassStages][R][128 B]

    // ---- phase 0 -----------------------------------------------------------
    // the token indices first, then what needs none: the first unit's A rows
    // (and x rows when dense) and the first expand tile's old out values
    int v_idx = 0;  // (ordered before the copies below by the asm)
    if (tid < T && ea.idx)
        asm volatile("ld.global.nc.b32 %0, [%1];\n" : "=r"(v_idx) : "l"(ea.idx + tid));
    int u = q0;
    if (u < n_units)
        issue_pass<E>(sa, u / S, u % S, kb, k1, 0, min(nst, kPassStages), true, dense, nullptr, 0,
                      T, sX, sA);
    cp_async_commit();
    int item = (int)blockIdx.x;
    FmaTile tt{};
    uint32_t old[8][2];
    if (item < n_items) {
        tt = fma_tile(ea, item, nchunks);
        fma_load_old<E, ADD>(ea, tt, old);
    }

    // token -> adapter map, and the tokens grouped by adapter in token order
    // (tokens without a LoRA term dropped)
    const int lt = tid < T && v_idx >= 0 && v_idx < L && clamp_rank(ea.ranks, v_idx, R) > 0 ? v_idx : -1;
    s_map[tid] = lt;
    int pos = 0;
    for (int lb = 0; lb < L; ++lb) {
        const unsigned m = __ballot_sync(0xffffffffu, lt == lb);
        if (lane == 0) s_wc[lb][warp] = __popc(m);
        if (lt == lb) pos = __popc(m & ((1u << lane) - 1u));
    }
    __syncthreads();
    if (tid == 0) {
        int run = 0;
        for (int lb = 0; lb < L; ++lb) {
            s_beg[lb] = run;
            int c = 0;
            for (int w = 0; w < kFThreads / 32; ++w) {
                const int v = s_wc[lb][w];
                s_wc[lb][w] = c;
                c += v;
            }
            s_cnt[lb] = c;
            run += c;
        }
    }
    __syncthreads();
    if (lt >= 0) s_tok[s_beg[lt] + s_wc[lt][warp] + pos] = tid;
    if (item < n_items && tid < kFRows) s_l[tid] = tt.t0 + tid < T ? s_map[tt.t0 + tid] : -1;
    // y rows of tokens without a LoRA term are zero (one CTA per row)
    for (int t = (int)blockIdx.x; t < T; t += (int)gridDim.x)
        if (s_map[t] < 0)
            for (int c = tid; c < W / 4; c += kFThreads)
                *reinterpret_cast<float4 *>(sa.y + (int64_t)t * sa.ldy + 4 * c) =
                    make_float4(0.f, 0.f, 0.f, 0.f);
    __syncthreads();  // s_tok, s_cnt complete
    if (!dense && u < n_units && s_cnt[u / S] > 0)
        issue_pass<E>(sa, u / S, u % S, kb, k1, 0, min(nst, kPassStages), false, true, s_tok,
                      s_beg[u / S], min(kSRows, s_cnt[u / S]), sX, sA);
    cp_async_commit();

    // ---- phase 1: shrink units (adapter, slice), K split over the cluster --
    // Every CTA of a cluster has the same units and token groups, so the
    // cluster barriers below are reached by all of them.
    for (; u < n_units; u += nclusters) {
        const int l = u / S, s = u % S;
        const int rl = clamp_rank(sa.ranks, l, R);
        const int ntok = s_cnt[l];
        const int rows_total = dense ? T : ntok;
        for (int g0 = 0; ntok > 0 && g0 < rows_total; g0 += kSRows) {
            const int cnt = min(kSRows, rows_total - g0);
            // warps over (m-tile, n-tile) tiles; with fewer than 8 tiles the
            // warps also split the stages (kpart = stage mod ksplit)
            const int m_t = (cnt + 15) / 16, tiles = m_t * RK8;
            const int ksplit = tiles >= 8 ? 1 : 8 / tiles;
            const int kpart = tiles >= 8 ? 0 : warp / tiles;
            const int tile0 = tiles >= 8 ? warp : warp % tiles;
            const bool busy = warp < tiles * ksplit;
            float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
            for (int p = 0; p < npass; ++p) {
                const int st0 = p * kPassStages, st1 = min(nst, st0 + kPassStages);
                if (u != q0 || g0 != 0 || p != 0) {  // (that pass was requested in phase 0)
                    __syncthreads();  // the stages are free
                    issue_pass<E>(sa, l, s, kb, k1, st0, st1, npass > 1 || g0 == 0, true,
                                  dense ? nullptr : s_tok, dense ? g0 : s_beg[l] + g0, cnt, sX, sA);
                    cp_async_commit();
                }
                cp_async_wait<0>();
                __syncthreads();
                if (busy) {
                    for (int st = st0 + kpart; st < st1; st += ksplit) {
                        const uint32_t xb = smem_u32(sX + (st - st0) * kSRows * 128);
                        const uint32_t ab = smem_u32(sA + (st - st0) * R * 128);
#pragma unroll
                        for (int kk = 0; kk < kSK / 16; ++kk) {
#pragma unroll
                            for (int j = 0; j < 2; ++j) {
                                const int tile = tile0 + 8 * j;
                                if (j == 0 || tile < tiles) {
                                    const int mt = tile / RK8, nt = tile - mt * RK8;
                                    uint32_t af[4], bf[2];
                                    ldmatrix_x4(af, xb + stage_off(mt * 16 + (lane & 15),
                                                                   2 * kk + (lane >> 4)));
                                    ldmatrix_x2(bf, ab + stage_off(nt * 8 + (lane & 7),
                                                                   2 * kk + ((lane >> 3) & 1)));
                                    mma16816<E>(acc[j], af, bf[0], bf[1]);
                                }
                            }
                        }
                    }
                }
            }
            // the warps' partials, then their sum (fixed order) to the row's
            // owner: row r goes to CTA r / 8, slot r % 8
            if (busy) {
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    const int tile = tile0 + 8 * j;
                    if (j == 0 || tile < tiles) {
                        const int mt = tile / RK8, nt = tile - mt * RK8;
                        const int r = kpart * m_t * 16 + mt * 16 + (lane >> 2);
                        const int c = nt * 8 + 2 * (lane & 3);
                        *reinterpret_cast<float2 *>(&s_part[r][c]) = make_float2(acc[j][0], acc[j][1]);
                        *reinterpret_cast<float2 *>(&s_part[r + 8][c]) = make_float2(acc[j][2], acc[j][3]);
                    }
                }
            }
            __syncthreads();
            for (int v = tid; v < cnt * (RK / 4); v += kFThreads) {
                const int r = v / (RK / 4), c = 4 * (v - r * (RK / 4));
                float4 sum = *reinterpret_cast<const float4 *>(&s_part[r][c]);
                for (int k = 1; k < ksplit; ++k) {
                    const float4 q = *reinterpret_cast<const float4 *>(&s_part[k * m_t * 16 + r][c]);
                    sum.x += q.x; sum.y += q.y; sum.z += q.z; sum.w += q.w;
                }
                st_cluster_v4(cluster_map(smem_u32(&s_recv[cr][r % 8][c]), r / 8), sum);
            }
            cluster_arrive();
            cluster_wait();
            // this CTA's rows: the CTAs' partials summed in CTA order, then y
            for (int v = tid; v < (kSRows / kCK) * RK; v += kFThreads) {
                const int i = v / RK, c = v - i * RK;
                const int r = cr * (kSRows / kCK) + i;
                if (r < cnt) {
                    const int t = dense ? g0 + r : s_tok[s_beg[l] + g0 + r];
                    if (!dense || s_map[t] == l) {
                        float sum = 0.f;
#pragma unroll
                        for (int src = 0; src < kCK; ++src) sum += s_recv[src][i][c];
                        sa.y[(int64_t)t * sa.ldy + s * R + c] = c < rl ? sa.scale * sum : 0.f;
                    }
                }
            }
            // the receive slots are written again only after every owner has
            // read them (the last round needs no barrier: no CTA exits before
            // the grid barrier)
            const bool more = g0 + kSRows < rows_total || u + nclusters < n_units;
            if (more) {
                cluster_arrive();
                cluster_wait();
            }
        }
    }
    // the first expand tile's B rows, in place of the shrink stages (no copy
    // into them may still be in flight: a unit without tokens never waited)
    cp_async_wait<0>();
    __syncthreads();
    if (item < n_items) fma_stage_b<E, RK8>(ea, tt, sB);
    cp_async_commit();
    grid.sync();  // (orders every thread's y stores before the reads below)

    // ---- phase 2: expand tiles ---------------------------------------------
    for (; item < n_items; item += (int)gridDim.x) {
        if (item != (int)blockIdx.x) {
            __syncthreads();  // the previous tile's shared memory is free
            tt = fma_tile(ea, item, nchunks);
            fma_stage_b<E, RK8>(ea, tt, sB);
            fma_load_old<E, ADD>(ea, tt, old);
            if (tid < kFRows) s_l[tid] = tt.t0 + tid < T ? s_map[tt.t0 + tid] : -1;
        }
        fma_stage_y<RK8>(ea, tt, s_y);
        cp_async_commit();
        cp_async_wait<0>();
        __syncthreads();
        fma_finish<E, ADD, RK8>(ea, tt, sB, s_y, s_l, old);
    }
}

using FusedFn = void (*)(const BgmvShrinkArgs, const BgmvExpandArgs, int, int);
template <typename E, bool ADD>
FusedFn fused_fn(int rk8) {
    switch (rk8) {
        case 1: return bgmv_fused_kernel<E, ADD, 1>;
        case 2: return bgmv_fused_kernel<E, ADD, 2>;
        case 3: return bgmv_fused_kernel<E, ADD, 3>;
        default: return bgmv_fused_kernel<E, ADD, 4>;
    }
}
FusedFn fused_fn(int dt, bool add, int rk8) {
    if (dt == LORA_F16) return add ? fused_fn<__half, true>(rk8) : fused_fn<__half, false>(rk8);
    return add ? fused_fn<__nv_bfloat16, true>(rk8) : fused_fn<__nv_bfloat16, false>(rk8);
}

constexpr int kFusedMaxSmem = fused_smem_bytes(LORA_BGMV_MAX_ADAPTERS, 4);
int g_fused_clusters = 0;  // clusters of kCK CTAs launched (one CTA per SM)

}  // namespace

cudaError_t configure_fused_kernels(const DeviceInfo &dev) {
    // clusters that fit at once for the largest variant, at most one CTA per SM
    int ncl = dev.sm_count / kCK;
    cudaError_t e = cudaSuccess;
    for (int dt = 0; dt < 2 && e == cudaSuccess; ++dt)
        for (int add = 0; add < 2 && e == cudaSuccess; ++add)
            for (int rk8 = 1; rk8 <= 4 && e == cudaSuccess; ++rk8) {
                const FusedFn fn = fused_fn(dt == 0 ? LORA_F16 : LORA_BF16, add != 0, rk8);
                e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, kFusedMaxSmem);
                if (e != cudaSuccess) break;
                cudaLaunchConfig_t cfg = {};
                cfg.gridDim = dim3((unsigned)(ncl > 0 ? ncl : 1) * kCK);
                cfg.blockDim = dim3(kFThreads);
                cfg.dynamicSmemBytes = kFusedMaxSmem;
                cudaLaunchAttribute attr[2];
                attr[0].id = cudaLaunchAttributeCooperative;
                attr[0].val.cooperative = 1;
                attr[1].id = cudaLaunchAttributeClusterDimension;
                attr[1].val.clusterDim.x = kCK;
                attr[1].val.clusterDim.y = 1;
                attr[1].val.clusterDim.z = 1;
                cfg.attrs = attr;
                cfg.numAttrs = 2;
                int active = 0;
                e = cudaOccupancyMaxActiveClusters(&active, fn, &cfg);
                if (e == cudaSuccess) ncl = std::min(ncl, active);
            }
    g_fused_clusters = e == cudaSuccess ? ncl : 0;
    return e;
}

const char *bgmv_fused_supported(const BgmvShrinkArgs &s, const BgmvExpandArgs &e) {
    if (g_fused_clusters < 1) return "the one-launch kernel's clusters do not fit on this device";
    if (s.T > kFusedMaxT) return "more than 256 tokens (use lora_bgmv_shrink_expand_slice)";
    if (s.R > kFusedMaxRank) return "R above 32 (use lora_bgmv_shrink_expand_slice)";
    if (s.add) return "the one-launch kernel writes y; it does not add to it";
    if (e.y_slice_stride != s.R) return "y slices must be packed (y_slice_stride == R)";
    return nullptr;
}

cudaError_t launch_bgmv_fused(lora_dtype_t dt, const BgmvShrinkArgs &sa, const BgmvExpandArgs &ea_in,
                              const DeviceInfo &dev, cudaStream_t stream) {
    if (sa.T == 0) return cudaSuccess;
    BgmvExpandArgs ea = ea_in;
    const int nchunks = fma_set_chunks(ea);
    const int n_items = ((sa.T + kFRows - 1) / kFRows) * nchunks;
    const int rk8 = (sa.R + 7) / 8;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(g_fused_clusters * kCK));
    cfg.blockDim = dim3(kFThreads);
    cfg.dynamicSmemBytes = (size_t)fused_smem_bytes(ea.idx ? ea.L : 1, rk8);
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = kCK;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, fused_fn(dt, ea.add != 0, rk8), sa, ea, nchunks, n_items);
}

}  // namespace lora
