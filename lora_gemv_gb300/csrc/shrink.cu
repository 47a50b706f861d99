// Shrink: y[t, s*R + i] (+)= scale * sum_h x[t, h] * A[l, s*R + i, h]   (i < r_l)
//
// Pages: vLLM PR #15655 summary (the kernel split into shrink and expand
// variants); vLLM PR #11579 (bgmv_shrink / sgmv_shrink, the fp32 rank
// buffer, and split-K shrink whose partial results are added); Punica issue
// #17 (tokens of one adapter share its weights; ranks are not limited to
// bins of 16/32/64).
//
// Design (GB300): per plan tile (<= 64 tokens of one adapter) the CTA
// computes Y[64, rows] = X[64, H] . A_l[rows, H]^T on the tensor cores
// (mma.sync m16n8k16, fp32 accumulate), where rows are the adapter's
// S * r_l live rows only (rank-aware: padded rows are never read).
//  - H is split across a thread-block CLUSTER of up to 16 CTAs (split-K);
//    each CTA streams its H range through a 4-stage cp.async pipeline
//    (x rows gathered through the plan's token order, A_l rows contiguous)
//    into 128-byte-swizzled shared memory;
//  - the partial tiles are reduced through distributed shared memory in a
//    fixed rank order (deterministic, no global scratch, no atomics), each
//    CTA of the cluster finishing a share of the rows;
//  - tiles of adapter -1 load nothing (block skipping); their y rows are
//    zeroed unless add_inputs.
#include <cooperative_groups.h>

#include <algorithm>

#include "common.cuh"
#include "kernels.h"

namespace cg = cooperative_groups;

namespace lora {
namespace {

constexpr int kThreads = 128;  // 4 warps, 16 token rows each
constexpr int kRows = 128;     // compacted A rows per CTA (grid.z covers more)
constexpr int kK = 64;         // H elements per pipeline stage (128 bytes)
constexpr int kStages = 4;
constexpr int kRedPitch = kRows + 4;  // floats per reduction row
constexpr int kSmem = kStages * (kTile + kRows) * kK * 2;  // largest configuration
// Shared memory for A tiles of `rows_cap` rows (a multiple of 16, <= kRows).
__host__ __device__ constexpr int smem_bytes(int rows_cap) {
    return kStages * (kTile + rows_cap) * kK * 2;
}
static_assert(kTile * kRedPitch * 4 <= smem_bytes(16), "reduction buffer fits in the stage buffers");

// 128-byte rows, 16-byte chunks XOR-swizzled by the row index.
__device__ __forceinline__ int swz(int row, int chunk) { return row * kK + ((chunk ^ (row & 7)) << 3); }

template <typename E, bool VEC>
__device__ __forceinline__ void load_stage(E *sX, E *sA, const E *__restrict__ x, int64_t ldx,
                                           const E *__restrict__ Al, int H, const int *s_rows,
                                           const int *s_arow, int n, int nrows, int h0, int h_end) {
    // x tile: n rows x 8 chunks
    for (int it = threadIdx.x; it < n * 8; it += kThreads) {
        const int r = it >> 3, c = it & 7;
        const int h = h0 + c * 8;
        const int row = s_rows[r];
        E *dst = sX + swz(r, c);
        if (VEC) {
            const bool ok = row >= 0 && h < h_end;
            const E *src = ok ? x + (int64_t)row * ldx + h : x;
            cp_async16(smem_u32(dst), src, ok ? 16 : 0);
        } else {
            uint4 v = make_uint4(0, 0, 0, 0);
            uint16_t *hv = reinterpret_cast<uint16_t *>(&v);
            if (row >= 0) {
                const uint16_t *src = reinterpret_cast<const uint16_t *>(x + (int64_t)row * ldx);
                for (int k = 0; k < 8; ++k)
                    if (h + k < h_end) hv[k] = __ldg(src + h + k);
            }
            *reinterpret_cast<uint4 *>(dst) = v;
        }
    }
    // A tile: nrows rows x 8 chunks (row = compacted live row of the adapter)
    for (int it = threadIdx.x; it < nrows * 8; it += kThreads) {
        const int r = it >> 3, c = it & 7;
        const int h = h0 + c * 8;
        const E *arow = Al + (int64_t)s_arow[r] * H;
        E *dst = sA + swz(r, c);
        if (VEC) {
            const bool ok = h < h_end;
            cp_async16(smem_u32(dst), ok ? arow + h : arow, ok ? 16 : 0);
        } else {
            uint4 v = make_uint4(0, 0, 0, 0);
            uint16_t *hv = reinterpret_cast<uint16_t *>(&v);
            const uint16_t *src = reinterpret_cast<const uint16_t *>(arow);
            for (int k = 0; k < 8; ++k)
                if (h + k < h_end) hv[k] = __ldg(src + h + k);
            *reinterpret_cast<uint4 *>(dst) = v;
        }
    }
}

template <typename E, bool VEC>
__global__ void __launch_bounds__(kThreads)
shrink_kernel(const ShrinkArgs a, int kchunk, int rows_cap) {
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ int s_rows[kTile];
    __shared__ int s_arow[kRows];

    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int g = lane >> 2, q = lane & 3;
    const int kc = blockIdx.x, ksplit = gridDim.x, rc = blockIdx.z;
    cg::cluster_group cluster = cg::this_cluster();

    // Every CTA of a cluster takes the same branch: the plan check reads the
    // same words, and the tile loop depends only on blockIdx.y / blockIdx.z.
    // The plan header and this CTA's first tile are read together.
    const int4 h0 = __ldcg(reinterpret_cast<const int4 *>(a.hdr));      // magic, T, L, kind
    const int4 h1 = __ldcg(reinterpret_cast<const int4 *>(a.hdr) + 1);  // nactive, ngroups, ntiles
    int4 tl_next = (int)blockIdx.y < a.max_tiles ? __ldcg(a.tiles + blockIdx.y)
                                                 : make_int4(-1, 0, 0, -1);
    if (h0.x != LORA_PLAN_MAGIC || h0.y != a.T || h0.z != a.L) {
        if (blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0 && threadIdx.x == 0)
            atomicOr(a.hdr + LORA_HDR_ERR, LORA_PLANERR_MISMATCH);
        return;
    }

    const E *__restrict__ x = static_cast<const E *>(a.x);
    const int H = a.H, R = a.R, S = a.S;
    const int h_begin = kc * kchunk;
    const int h_end = min(H, h_begin + kchunk);
    const int nsteps = h_end > h_begin ? (h_end - h_begin + kK - 1) / kK : 0;
    E *sX = reinterpret_cast<E *>(smem);
    E *sA = sX + kStages * kTile * kK;
    float *sRed = reinterpret_cast<float *>(smem);

    const int n_tiles = min(h1.z, a.max_tiles);
    for (int tile = blockIdx.y; tile < n_tiles; tile += gridDim.y) {
        const int4 tl = tl_next;
        if (tile + (int)gridDim.y < n_tiles) tl_next = __ldcg(a.tiles + tile + gridDim.y);
        const int l = tl.x, p0 = tl.y, n = tl.z;
        const int rl = l >= 0 && l < a.L ? clamp_rank(a.ranks, l, R) : 0;

        // y columns that get no term: every column of inactive tokens, the
        // columns i >= r_l of each slice otherwise.  Written by one CTA.
        if (!a.add && kc == 0 && rc == 0 && rl < R) {
            for (int it = threadIdx.x; it < n * S * R; it += kThreads) {
                const int i = it / (S * R), j = it % (S * R);
                if (j % R < rl) continue;
                const int row = a.perm[p0 + i];
                if (row >= 0 && row < a.T) a.y[(int64_t)row * a.ldy + j] = 0.f;
            }
        }
        const int row0 = rc * kRows;
        const int nrows = min(kRows, S * rl - row0);
        if (nrows <= 0) continue;

        if (threadIdx.x < kTile) {
            int row = -1;
            if (threadIdx.x < n) {
                row = __ldcg(a.perm + p0 + threadIdx.x);
                if (row < 0 || row >= a.T) row = -1;
            }
            s_rows[threadIdx.x] = row;
        }
        if (threadIdx.x < kRows) {
            const int c = row0 + threadIdx.x;
            s_arow[threadIdx.x] = threadIdx.x < nrows ? (c / rl) * R + c % rl : 0;
        }
        __syncthreads();

        const E *Al = static_cast<const E *>(a.A) + (int64_t)l * S * R * H;
        const int NT = (nrows + 7) / 8;
        const bool wact = warp * 16 < n;

        float acc[16][4];
#pragma unroll
        for (int i = 0; i < 16; ++i)
#pragma unroll
            for (int k = 0; k < 4; ++k) acc[i][k] = 0.f;

#pragma unroll
        for (int st = 0; st < kStages - 1; ++st) {
            if (st < nsteps)
                load_stage<E, VEC>(sX + st * kTile * kK, sA + st * rows_cap * kK, x, a.ldx, Al, H,
                                   s_rows, s_arow, n, nrows, h_begin + st * kK, h_end);
            cp_async_commit();
        }
        for (int step = 0; step < nsteps; ++step) {
            cp_async_wait<kStages - 2>();
            __syncthreads();
            const int nxt = step + kStages - 1;
            if (nxt < nsteps) {
                const int b = nxt % kStages;
                load_stage<E, VEC>(sX + b * kTile * kK, sA + b * rows_cap * kK, x, a.ldx, Al, H,
                                   s_rows, s_arow, n, nrows, h_begin + nxt * kK, h_end);
            }
            cp_async_commit();
            if (wact) {
                const int b = step % kStages;
                const E *bx = sX + b * kTile * kK;
                const E *ba = sA + b * rows_cap * kK;
#pragma unroll
                for (int kk = 0; kk < kK / 16; ++kk) {
                    uint32_t af[4];
                    const int ar = warp * 16 + (lane & 7) + 8 * ((lane >> 3) & 1);
                    ldmatrix_x4(af, smem_u32(bx + swz(ar, 2 * kk + (lane >> 4))));
#pragma unroll
                    for (int np = 0; np < 8; ++np) {
                        if (2 * np < NT) {
                            uint32_t bf[4];
                            const int br = 8 * (2 * np + (lane >> 4)) + (lane & 7);
                            ldmatrix_x4(bf, smem_u32(ba + swz(br, 2 * kk + ((lane >> 3) & 1))));
                            mma16816<E>(acc[2 * np], af, bf[0], bf[1]);
                            if (2 * np + 1 < NT) mma16816<E>(acc[2 * np + 1], af, bf[2], bf[3]);
                        }
                    }
                }
            }
        }
        cp_async_wait<0>();
        __syncthreads();

        // partial tile -> own shared memory
        if (wact) {
#pragma unroll
            for (int nt = 0; nt < 16; ++nt) {
                if (nt < NT) {
                    const int r0 = warp * 16 + g, c0 = nt * 8 + 2 * q;
                    sRed[r0 * kRedPitch + c0] = acc[nt][0];
                    sRed[r0 * kRedPitch + c0 + 1] = acc[nt][1];
                    sRed[(r0 + 8) * kRedPitch + c0] = acc[nt][2];
                    sRed[(r0 + 8) * kRedPitch + c0 + 1] = acc[nt][3];
                }
            }
        }
        if (ksplit > 1) cluster.sync();
        else __syncthreads();

        // fixed-order reduction over the cluster; CTA kc finishes rows i = kc (mod ksplit)
        const int my_rows = n > kc ? (n - kc + ksplit - 1) / ksplit : 0;
        for (int it = threadIdx.x; it < my_rows * nrows; it += kThreads) {
            const int i = kc + ksplit * (it / nrows), c = it % nrows;
            const int row = s_rows[i];
            // all ranks' partials are loaded at once, then added in rank order
            float part[16];
#pragma unroll
            for (int r = 0; r < 16; ++r) {
                part[r] = 0.f;
                if (r < ksplit) {
                    const float *src = ksplit > 1 ? cluster.map_shared_rank(sRed, r) : sRed;
                    part[r] = src[i * kRedPitch + c];
                }
            }
            float sum = 0.f;
#pragma unroll
            for (int r = 0; r < 16; ++r)
                if (r < ksplit) sum += part[r];
            if (row >= 0) {
                float *yp = a.y + (int64_t)row * a.ldy + s_arow[c];
                const float v = a.scale * sum;
                *yp = a.add ? *yp + v : v;
            }
        }
        if (ksplit > 1) cluster.sync();
        else __syncthreads();
    }
}

template <typename E, bool VEC>
cudaError_t configure_one(int max_cluster) {
    cudaError_t e = cudaFuncSetAttribute(shrink_kernel<E, VEC>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    if (e != cudaSuccess) return e;
    if (max_cluster > 8)
        e = cudaFuncSetAttribute(shrink_kernel<E, VEC>,
                                 cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    return e;
}

template <typename E>
cudaError_t launch_dtype(const ShrinkArgs &a, bool vec, int ksplit, int kchunk, int rows_cap,
                         dim3 grid, cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem_bytes(rows_cap);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = ksplit;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (vec) return cudaLaunchKernelEx(&cfg, shrink_kernel<E, true>, a, kchunk, rows_cap);
    return cudaLaunchKernelEx(&cfg, shrink_kernel<E, false>, a, kchunk, rows_cap);
}

}  // namespace

cudaError_t configure_shrink_kernels(DeviceInfo *info) {
    // Largest cluster the pool can hold with this kernel's shared memory.
    int max_cluster = 8;
    {
        cudaError_t e = cudaFuncSetAttribute(shrink_kernel<__half, true>,
                                             cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e == cudaSuccess) e = cudaFuncSetAttribute(shrink_kernel<__half, true>,
                                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                       kSmem);
        if (e != cudaSuccess) return e;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(16, 1, 1);
        cfg.blockDim = dim3(kThreads);
        cfg.dynamicSmemBytes = kSmem;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 16;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, shrink_kernel<__half, true>, &cfg) == cudaSuccess &&
            n > 0)
            max_cluster = 16;
        cudaGetLastError();  // a refused query is not an error: fall back to 8
    }
    info->max_cluster = max_cluster;
    cudaError_t e;
    if ((e = configure_one<__half, true>(max_cluster)) != cudaSuccess) return e;
    if ((e = configure_one<__half, false>(max_cluster)) != cudaSuccess) return e;
    if ((e = configure_one<__nv_bfloat16, true>(max_cluster)) != cudaSuccess) return e;
    return configure_one<__nv_bfloat16, false>(max_cluster);
}

cudaError_t launch_shrink(lora_dtype_t dt, const ShrinkArgs &a, const DeviceInfo &dev,
                          cudaStream_t stream) {
    if (a.T == 0) return cudaSuccess;
    const bool vec = (reinterpret_cast<uintptr_t>(a.x) & 15) == 0 &&
                     (reinterpret_cast<uintptr_t>(a.A) & 15) == 0 && a.ldx % 8 == 0 &&
                     a.H % 8 == 0;
    // Tile slots: see launch_expand.  CTAs loop over any further tiles.
    const long long est = (a.T + kTile - 1) / kTile + (long long)std::min(a.L, a.T) + 1;
    const int gy = (int)std::max<long long>(1, std::min<long long>({est, a.max_tiles, 65535}));
    const int gz = (a.S * a.R + kRows - 1) / kRows;
    const int rows_cap = std::min(kRows, (a.S * a.R + 15) / 16 * 16);
    // CTAs resident per SM (shared memory, and 128 registers x 128 threads)
    const int per_sm = std::max(1, std::min(4, (227 * 1024) / (smem_bytes(rows_cap) + 1024)));
    // Split K across a cluster so that the grid fills the resident slots,
    // each CTA keeping >= 2 pipeline stages of work.
    const int target = per_sm * dev.sm_count;
    int ksplit = 1;
    while (ksplit < dev.max_cluster && (long long)gy * gz * ksplit * 2 <= target &&
           (a.H + ksplit * 2 * kK - 1) / (ksplit * 2 * kK) >= 2)
        ksplit *= 2;
    int kchunk = ((a.H + ksplit - 1) / ksplit + kK - 1) / kK * kK;
    while (ksplit > 1 && (long long)(ksplit - 1) * kchunk >= a.H) ksplit /= 2;  // no empty CTAs
    kchunk = ((a.H + ksplit - 1) / ksplit + kK - 1) / kK * kK;
    dim3 grid(ksplit, gy, gz);
    return dt == LORA_F16 ? launch_dtype<__half>(a, vec, ksplit, kchunk, rows_cap, grid, stream)
                          : launch_dtype<__nv_bfloat16>(a, vec, ksplit, kchunk, rows_cap, grid, stream);
}

}  // namespace lora
