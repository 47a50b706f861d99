// Fused shrink + expand_slice for one batch: one thread-block cluster per plan
// tile (<= 64 tokens of one adapter).
//
// Pages: vLLM PR #15655 (shrink and expand variants of the LoRA kernel);
// vLLM PR #11579 (the fp32 rank buffer between them, split-K shrink adding
// partials, expand_slice over the slices of a fused output, add_inputs).
// The shrink result is identical in meaning to lora_shrink (y is written);
// fusing only removes a launch, a dependency gap and the re-read of y from
// HBM, which dominate at decode batch sizes.
//
// Per cluster of C CTAs (8 warps each):
//  1. shrink: CTA c takes H range c of C; its warps split that range again
//     (and the tile's m16 blocks).  x rows and the adapter's live A rows are
//     read with 16-byte loads straight into mma.sync fragments (the
//     contraction index is permuted so each thread's 8 consecutive h fill
//     two 16-wide k steps);
//  2. partials: warp partials are summed in shared memory (fixed order),
//     then across the cluster through distributed shared memory, each CTA
//     finishing a 1/C share of the tile and writing it to y (fp32);
//  3. after a cluster barrier (release/acquire at cluster scope) every CTA
//     reads the finished y rows from L2 and expands its 1/C share of the
//     32-column blocks of all slices (warp units as in the warp-streaming
//     expand: B fragments and out rows from HBM with 16-byte accesses).
#include <cooperative_groups.h>

#include <algorithm>

#include "common.cuh"
#include "frag.cuh"
#include "kernels.h"

namespace cg = cooperative_groups;

namespace lora {
namespace {

constexpr int kFThreads = 256;
constexpr int kFWarps = kFThreads / 32;
constexpr int kFCols = 32;  // output columns per expand unit

__host__ __device__ constexpr int part_pitch(int ntmax) { return ntmax * 8 + 4; }
__host__ __device__ constexpr int fused_smem(int ntmax) {
    return (kFWarps * 16 + kTile) * part_pitch(ntmax) * (int)sizeof(float);
}

// Two CTAs per SM for the small register footprints (decode ranks), one above.
template <typename E, bool ADD, int NTMAX, int KSMAX>
__global__ void __launch_bounds__(kFThreads, (NTMAX * KSMAX <= 8 ? 2 : 1))
fused_kernel(const FusedArgs a, int hchunk, int y_vec) {
    extern __shared__ __align__(16) float fsm[];
    __shared__ int s_rows[kTile];
    constexpr int PP = part_pitch(NTMAX);
    float *P = fsm;                        // [kFWarps][16][PP] warp partials
    float *Ct = fsm + kFWarps * 16 * PP;   // [64][PP] CTA partial of the tile

    cg::cluster_group cluster = cg::this_cluster();
    const int csize = gridDim.x, c = blockIdx.x;  // one cluster = one row of the grid
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int g = lane >> 2, q = lane & 3;

    // Every CTA of a cluster takes the same branches below: they read the
    // same plan words and share blockIdx.y.
    const int4 h0 = __ldg(reinterpret_cast<const int4 *>(a.hdr));
    const int4 h1 = __ldg(reinterpret_cast<const int4 *>(a.hdr) + 1);
    int4 tl_next = (int)blockIdx.y < a.max_tiles ? __ldg(a.tiles + blockIdx.y)
                                                 : make_int4(-1, 0, 0, -1);
    if (h0.x != LORA_PLAN_MAGIC || h0.y != a.T || h0.z != a.L) {
        if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0)
            atomicOr(a.hdr + LORA_HDR_ERR, LORA_PLANERR_MISMATCH);
        return;
    }
    const int n_tiles = min(h1.z, a.max_tiles);
    const E *__restrict__ x = static_cast<const E *>(a.x);
    E *__restrict__ out = static_cast<E *>(a.out);
    const int H = a.H, R = a.R, S = a.S;
    const int ncb = a.cb_begin[a.num_slices];

    for (int tile = blockIdx.y; tile < n_tiles; tile += gridDim.y) {
        const int4 tl = tl_next;
        if (tile + (int)gridDim.y < n_tiles) tl_next = __ldg(a.tiles + tile + gridDim.y);
        const int l = tl.x, n = tl.z;
        const int rl = l >= 0 && l < a.L ? clamp_rank(a.ranks, l, R) : 0;

        if (threadIdx.x < kTile) {
            int row = __ldg(a.tile_rows + (int64_t)tile * kTile + threadIdx.x);
            s_rows[threadIdx.x] = row >= a.T ? -1 : row;
        }
        __syncthreads();

        // y columns without a term: all of an inactive row, ranks >= r_l otherwise
        if (rl < R) {
            for (int it = threadIdx.x + c * kFThreads; it < n * S * R; it += csize * kFThreads) {
                const int i = it / (S * R), j = it - i * (S * R);
                const int row = s_rows[i];
                if (j % R >= rl && row >= 0) a.y[(int64_t)row * a.ldy + j] = 0.f;
            }
        }
        if (rl == 0) {  // adapter -1 / rank 0: out untouched with add_inputs, zeros without
            if (!ADD) {
                for (int it = threadIdx.x; it < n * ncb * 4; it += kFThreads) {
                    const int i = it / (ncb * 4), r2 = it - i * (ncb * 4);
                    const int b = r2 >> 2, part = r2 & 3;
                    if (b % csize != c) continue;
                    int s = 0;
                    while (s + 1 < a.num_slices && b >= a.cb_begin[s + 1]) ++s;
                    const int cc = (b - a.cb_begin[s]) * kFCols + 8 * part;
                    const int row = s_rows[i];
                    if (row >= 0 && cc < a.N[s])
                        st_global_v4(out + (int64_t)row * a.ldo + a.off[s] + cc, make_uint4(0, 0, 0, 0));
                }
            }
            __syncthreads();
            continue;
        }

        // ---------------- 1. shrink partials
        const int SR = S * rl;  // live A rows (<= NTMAX * 8, checked by the host)
        const int NT = (SR + 7) / 8;
        const int nmb = (n + 15) / 16;
        const int nmbp = nmb <= 1 ? 1 : (nmb <= 2 ? 2 : 4);
        const int kparts = kFWarps / nmbp;
        const int mb = warp % nmbp, kp = warp / nmbp;
        const int hc0 = c * hchunk, hc1 = min(H, hc0 + hchunk);
        const int steps = hc1 > hc0 ? (hc1 - hc0 + 31) / 32 : 0;
        const int st0 = steps * kp / kparts, st1 = steps * (kp + 1) / kparts;

        float acc[NTMAX][4];
#pragma unroll
        for (int i = 0; i < NTMAX; ++i)
#pragma unroll
            for (int k = 0; k < 4; ++k) acc[i][k] = 0.f;
        if (mb < nmb) {
            const int r0 = s_rows[mb * 16 + g], r1 = s_rows[mb * 16 + g + 8];
            const E *x0 = x + (int64_t)(r0 < 0 ? 0 : r0) * a.ldx;
            const E *x1 = x + (int64_t)(r1 < 0 ? 0 : r1) * a.ldx;
            const E *Al = static_cast<const E *>(a.A) + (int64_t)l * S * R * H;
            int aoff[NTMAX];  // A row of this thread's n-tile row, -1 past the live rows
#pragma unroll
            for (int nt = 0; nt < NTMAX; ++nt) {
                const int cr = nt * 8 + g;
                aoff[nt] = cr < SR ? (cr / rl) * R + cr % rl : -1;
            }
            for (int st = st0; st < st1; ++st) {
                const int h = hc0 + st * 32 + 8 * q;
                const bool hv = h < hc1;
                const uint4 z = make_uint4(0, 0, 0, 0);
                const uint4 xa = (hv && r0 >= 0) ? __ldg(reinterpret_cast<const uint4 *>(x0 + h)) : z;
                const uint4 xb = (hv && r1 >= 0) ? __ldg(reinterpret_cast<const uint4 *>(x1 + h)) : z;
                uint4 av[NTMAX];
#pragma unroll
                for (int nt = 0; nt < NTMAX; ++nt)
                    av[nt] = (nt < NT && hv && aoff[nt] >= 0)
                                 ? __ldg(reinterpret_cast<const uint4 *>(Al + (int64_t)aoff[nt] * H + h))
                                 : z;
#pragma unroll
                for (int kk = 0; kk < 2; ++kk) {
                    const uint32_t af[4] = {kk ? xa.z : xa.x, kk ? xb.z : xb.x, kk ? xa.w : xa.y,
                                            kk ? xb.w : xb.y};
#pragma unroll
                    for (int nt = 0; nt < NTMAX; ++nt)
                        if (nt < NT)
                            mma16816<E>(acc[nt], af, kk ? av[nt].z : av[nt].x,
                                        kk ? av[nt].w : av[nt].y);
                }
            }
        }
        // warp partials -> P[warp]
        if (mb < nmb) {
            float *pw = P + warp * 16 * PP;
#pragma unroll
            for (int nt = 0; nt < NTMAX; ++nt) {
                if (nt < NT) {
                    const int cc = nt * 8 + 2 * q;
                    pw[g * PP + cc] = acc[nt][0];
                    pw[g * PP + cc + 1] = acc[nt][1];
                    pw[(g + 8) * PP + cc] = acc[nt][2];
                    pw[(g + 8) * PP + cc + 1] = acc[nt][3];
                }
            }
        }
        __syncthreads();
        // CTA partial: sum over the warps that split this m16 block's H range
        for (int it = threadIdx.x; it < n * SR; it += kFThreads) {
            const int i = it / SR, j = it - i * SR;
            const int m = i >> 4, r = i & 15;
            float sum = 0.f;
            for (int k = 0; k < kparts; ++k) sum += P[((k * nmbp + m) * 16 + r) * PP + j];
            Ct[i * PP + j] = sum;
        }

        // ---------------- 2. cluster reduction -> y
        cluster.sync();
        {
            const int E_ = n * SR;
            const int e0 = (int)((long long)E_ * c / csize), e1 = (int)((long long)E_ * (c + 1) / csize);
            for (int it = e0 + threadIdx.x; it < e1; it += kFThreads) {
                const int i = it / SR, j = it - i * SR;
                float part[16];
#pragma unroll
                for (int r = 0; r < 16; ++r) {
                    part[r] = 0.f;
                    if (r < csize) part[r] = cluster.map_shared_rank(Ct, r)[i * PP + j];
                }
                float sum = 0.f;
#pragma unroll
                for (int r = 0; r < 16; ++r)
                    if (r < csize) sum += part[r];
                const int row = s_rows[i];
                if (row >= 0) a.y[(int64_t)row * a.ldy + (j / rl) * R + j % rl] = a.scale_s * sum;
            }
        }
        cluster.sync();  // y of the whole tile is written; no CTA reads remote shared memory after this

        // ---------------- 3. expand this CTA's column blocks
        const int KS = (rl + 15) / 16;
        const int nmp = (n + 31) / 32;  // 32-row pairs of m16 blocks
        const int nb_c = ncb > c ? (ncb - c + csize - 1) / csize : 0;
        int y_key = -1;
        uint32_t ah[2][KSMAX][4], al[2][KSMAX][4];
        float fscale[2][2];
        for (int u = warp; u < nmp * nb_c; u += kFWarps) {
            const int mp = u / nb_c, b = c + (u - mp * nb_c) * csize;
            int s = 0;
            while (s + 1 < a.num_slices && b >= a.cb_begin[s + 1]) ++s;
            const int c0 = (b - a.cb_begin[s]) * kFCols;
            const int Ns = a.N[s];
            const int64_t col = (int64_t)a.off[s] + c0 + 8 * q;
            const bool col_ok = c0 + 8 * q < Ns;
            int rows[2][2];
#pragma unroll
            for (int mm = 0; mm < 2; ++mm)
#pragma unroll
                for (int h = 0; h < 2; ++h) rows[mm][h] = s_rows[mp * 32 + mm * 16 + g + 8 * h];
            uint4 old[2][2];
            if (ADD && col_ok) {
#pragma unroll
                for (int mm = 0; mm < 2; ++mm)
#pragma unroll
                    for (int h = 0; h < 2; ++h)
                        if (rows[mm][h] >= 0)
                            old[mm][h] = ld_global_v4(out + (int64_t)rows[mm][h] * a.ldo + col);
            }
            uint2 bf[KSMAX][4];
            load_bfrags<E, KSMAX>(bf, static_cast<const E *>(a.B[s]) + (int64_t)l * Ns * R, Ns, R,
                                  c0, rl, KS, g, q);
            if (y_key != mp * LORA_MAX_SLICES + s) {
                y_key = mp * LORA_MAX_SLICES + s;
                build_yfrags<E, 2, KSMAX, true>(ah, al, fscale, rows, a.y + (int64_t)s * R, a.ldy,
                                                rl, KS, a.scale, y_vec != 0, q);
            }
#pragma unroll
            for (int mm = 0; mm < 2; ++mm) {
                if (mp * 32 + mm * 16 >= n) break;
                expand_block<E, ADD, KSMAX>(out, a.ldo, col, rows[mm], ah[mm], al[mm], bf,
                                            fscale[mm], old[mm], KS, col_ok);
            }
        }
        __syncthreads();  // s_rows and the partial buffers are reused by the next tile
    }
}

constexpr int kMaxCluster = 16;

template <typename E, bool ADD, int NTMAX, int KSMAX>
cudaError_t configure_one(bool nonportable) {
    cudaError_t e = cudaFuncSetAttribute(fused_kernel<E, ADD, NTMAX, KSMAX>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         fused_smem(NTMAX));
    if (e == cudaSuccess && nonportable)
        e = cudaFuncSetAttribute(fused_kernel<E, ADD, NTMAX, KSMAX>,
                                 cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    return e;
}

template <typename E, bool ADD>
cudaError_t configure_add(bool np) {
    cudaError_t e;
    if ((e = configure_one<E, ADD, 2, 1>(np)) != cudaSuccess) return e;
    if ((e = configure_one<E, ADD, 4, 1>(np)) != cudaSuccess) return e;
    if ((e = configure_one<E, ADD, 8, 1>(np)) != cudaSuccess) return e;
    if ((e = configure_one<E, ADD, 4, 2>(np)) != cudaSuccess) return e;
    if ((e = configure_one<E, ADD, 8, 2>(np)) != cudaSuccess) return e;
    if ((e = configure_one<E, ADD, 16, 2>(np)) != cudaSuccess) return e;
    if ((e = configure_one<E, ADD, 8, 4>(np)) != cudaSuccess) return e;
    return configure_one<E, ADD, 16, 4>(np);
}

template <typename E, bool ADD, int NTMAX, int KSMAX>
cudaError_t launch_one(const FusedArgs &a, int csize, int gy, int hchunk, int y_vec,
                       cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(csize, gy, 1);
    cfg.blockDim = dim3(kFThreads);
    cfg.dynamicSmemBytes = fused_smem(NTMAX);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = csize;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, fused_kernel<E, ADD, NTMAX, KSMAX>, a, hchunk, y_vec);
}

// (n-tile class, k-step class) instantiations: live A rows S*R <= 8*NTMAX and
// ranks R <= 16*KSMAX.
template <typename E, bool ADD>
cudaError_t launch_add(const FusedArgs &a, int csize, int gy, int hchunk, int y_vec,
                       cudaStream_t st) {
    const int nt = (a.S * a.R + 7) / 8, ks = (a.R + 15) / 16;
    if (ks <= 1) {
        if (nt <= 2) return launch_one<E, ADD, 2, 1>(a, csize, gy, hchunk, y_vec, st);
        if (nt <= 4) return launch_one<E, ADD, 4, 1>(a, csize, gy, hchunk, y_vec, st);
        return launch_one<E, ADD, 8, 1>(a, csize, gy, hchunk, y_vec, st);
    }
    if (ks <= 2) {
        if (nt <= 4) return launch_one<E, ADD, 4, 2>(a, csize, gy, hchunk, y_vec, st);
        if (nt <= 8) return launch_one<E, ADD, 8, 2>(a, csize, gy, hchunk, y_vec, st);
        return launch_one<E, ADD, 16, 2>(a, csize, gy, hchunk, y_vec, st);
    }
    if (nt <= 8) return launch_one<E, ADD, 8, 4>(a, csize, gy, hchunk, y_vec, st);
    return launch_one<E, ADD, 16, 4>(a, csize, gy, hchunk, y_vec, st);
}

int g_max_cluster = 8;

}  // namespace

cudaError_t configure_fused_kernels(const DeviceInfo &dev) {
    const bool np = dev.max_cluster > 8;
    g_max_cluster = dev.max_cluster;
    cudaError_t e;
    if ((e = configure_add<__half, false>(np)) != cudaSuccess) return e;
    if ((e = configure_add<__half, true>(np)) != cudaSuccess) return e;
    if ((e = configure_add<__nv_bfloat16, false>(np)) != cudaSuccess) return e;
    return configure_add<__nv_bfloat16, true>(np);
}

cudaError_t launch_fused(lora_dtype_t dt, const FusedArgs &a_in, const DeviceInfo &dev,
                         cudaStream_t stream) {
    FusedArgs a = a_in;
    // Shapes served: ranks <= 64, live rows S*R <= 128, 16-byte aligned rows
    // of x, A, out and B (else the caller runs shrink and expand_slice).
    bool ok = a.R <= 64 && a.S * a.R <= 128 && a.H % 8 == 0 && a.ldx % 8 == 0 && a.R % 8 == 0 &&
              a.ldo % 8 == 0 && (reinterpret_cast<uintptr_t>(a.x) & 15) == 0 &&
              (reinterpret_cast<uintptr_t>(a.A) & 15) == 0 &&
              (reinterpret_cast<uintptr_t>(a.out) & 15) == 0;
    for (int s = 0; s < a.num_slices; ++s)
        ok = ok && a.off[s] % 8 == 0 && a.N[s] % 8 == 0 &&
             (reinterpret_cast<uintptr_t>(a.B[s]) & 15) == 0;
    if (!ok) return cudaErrorNotSupported;
    if (a.T == 0) return cudaSuccess;
    a.cb_begin[0] = 0;
    for (int s = 0; s < a.num_slices; ++s)
        a.cb_begin[s + 1] = a.cb_begin[s] + (a.N[s] + kFCols - 1) / kFCols;
    for (int s = a.num_slices; s < LORA_MAX_SLICES; ++s) a.cb_begin[s + 1] = a.cb_begin[s];

    const long long est = (a.T + kTile - 1) / kTile + (long long)std::min(a.L, a.T) + 1;
    const int gy = (int)std::max<long long>(1, std::min<long long>({est, a.max_tiles, 65535}));
    // cluster size: enough CTAs to fill the GPU, H split into >= 256-wide pieces
    int csize = 1;
    while (csize < std::min(g_max_cluster, kMaxCluster) && (long long)gy * csize * 2 <= 2LL * dev.sm_count &&
           a.H / (csize * 2) >= 256)
        csize *= 2;
    const int hchunk = ((a.H + csize - 1) / csize + 31) / 32 * 32;
    const int y_vec = (reinterpret_cast<uintptr_t>(a.y) & 15) == 0 && a.ldy % 4 == 0 && a.R % 4 == 0;
    if (dt == LORA_F16)
        return a.add ? launch_add<__half, true>(a, csize, gy, hchunk, y_vec, stream)
                     : launch_add<__half, false>(a, csize, gy, hchunk, y_vec, stream);
    return a.add ? launch_add<__nv_bfloat16, true>(a, csize, gy, hchunk, y_vec, stream)
                 : launch_add<__nv_bfloat16, false>(a, csize, gy, hchunk, y_vec, stream);
}

}  // namespace lora
