// Token grouping: turns a BGMV per-token adapter index or an SGMV segment
// table into the plan every operator reads (token order, adapter groups and
// 64-token work tiles).
//
// Pages: Punica issue #17 "The smallest rank supported is 16?" (BGMV = one
// adapter per input, SGMV = segments of inputs sharing an adapter, the
// "AAABCC" batch); vLLM PR #15655 summary (cheap mask construction, blocks
// without work skipped): here the mask becomes a stable counting
// sort done once per batch on the device, and skipped blocks are simply the
// tiles that do not exist (empty adapters) or carry adapter -1.
//
// Both kernels run as ONE block of 1024 threads: the inputs are at most a few
// hundred KB of int32 and the result feeds every LoRA layer of a step.
#include <algorithm>

#include "common.cuh"
#include "kernels.h"

namespace lora {

namespace {

constexpr int kPlanThreads = 1024;
constexpr int kPlanWarps = kPlanThreads / 32;

// Cut groups [0, G) into tiles of <= kTile tokens, then the inactive tokens
// perm[n_active, T), and write each tile's token rows.  Group arrays must be
// visible to the whole block.  With perm_s / tiles_s (shared copies of perm
// and room for the tile records) the row lists are built from shared memory.
__device__ void emit_tiles(const PlanPtrs &p, int T, int n_active, int G, int *ws,
                           const int *perm_s = nullptr, int4 *tiles_s = nullptr) {
    int carry = 0;
    for (int base = 0; base < G; base += blockDim.x) {  // block-uniform loop
        const int g = base + threadIdx.x;
        const int cnt = g < G ? p.group_count[g] : 0;
        const int nt = (cnt + kTile - 1) / kTile;
        int total;
        const int ex = block_exclusive_scan(nt, ws, &total);
        if (g < G) {
            const int st = p.group_start[g], lo = p.group_lora[g];
            for (int k = 0; k < nt; ++k) {
                const int4 tr = make_int4(lo, st + k * kTile, min(kTile, cnt - k * kTile), g);
                p.tiles[carry + ex + k] = tr;
                if (tiles_s) tiles_s[carry + ex + k] = tr;
            }
        }
        carry += total;
    }
    const int n_in = T - n_active;
    const int nti = (n_in + kTile - 1) / kTile;
    for (int k = threadIdx.x; k < nti; k += blockDim.x) {
        const int p0 = n_active + k * kTile;
        const int4 tr = make_int4(-1, p0, min(kTile, T - p0), -1);
        p.tiles[carry + k] = tr;
        if (tiles_s) tiles_s[carry + k] = tr;
    }
    if (threadIdx.x == 0) p.hdr[LORA_HDR_NTILES] = carry + nti;
    // every tile's token rows, -1 past its count
    __syncthreads();
    const int ntl = carry + nti;
    for (int it = threadIdx.x; it < ntl * kTile; it += blockDim.x) {
        const int k = it / kTile, i = it - k * kTile;
        const int4 t = tiles_s ? tiles_s[k] : p.tiles[k];
        p.tile_rows[it] = i < t.z ? (perm_s ? perm_s[t.y + i] : p.perm[t.y + i]) : -1;
    }
}

__device__ void write_header(const PlanPtrs &p, int T, int L, int kind, int n_active, int G,
                             int bad, int err) {
    if (threadIdx.x == 0) {
        p.hdr[LORA_HDR_T] = T;
        p.hdr[LORA_HDR_L] = L;
        p.hdr[LORA_HDR_KIND] = kind;
        p.hdr[LORA_HDR_NACTIVE] = n_active;
        p.hdr[LORA_HDR_NGROUPS] = G;
        p.hdr[LORA_HDR_BAD_IDS] = bad;
        p.hdr[LORA_HDR_ERR] = err;
        for (int w = LORA_HDR_ERR + 1; w < LORA_HDR_WORDS; ++w) p.hdr[w] = 0;
        p.hdr[LORA_HDR_MAGIC] = LORA_PLAN_MAGIC;
    }
}

// ---------------------------------------------------------------- BGMV
// Stable counting sort.  Warp w owns a contiguous token range; pass 1 builds
// a private histogram per warp, a scan over (adapter, warp) gives every warp
// its first slot per adapter, pass 2 places tokens using match_any ranks so
// equal ids keep their token order.  Shared memory: kPlanWarps * L ints.
// STAGED (small batches): idx and perm live in shared memory (one coalesced
// read of idx, no dependent global reads afterwards); shared layout
// [kPlanWarps][L] histogram, idx[T], perm[T], tile records.
template <int NW, bool STAGED>
__global__ void __launch_bounds__(NW * 32, 1)
group_tokens_kernel(const int32_t *__restrict__ idx_g, int T, int L, PlanPtrs p) {
    constexpr int kPlanWarps = NW;
    extern __shared__ __align__(16) int hist[];  // [kPlanWarps][L]
    __shared__ int ws[40];
    __shared__ int s_inact[kPlanWarps];
    __shared__ int s_bad;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int *idx_s = hist + kPlanWarps * L;  // STAGED only
    // A programmatic dependent (the shrink) may be scheduled now: it reads
    // the plan only after its own wait, i.e. after this grid completes.
    grid_dep_wait();
    grid_dep_launch();
    int *perm_s = idx_s + T;
    // tile records start at a multiple of 4 ints (16 bytes): kPlanWarps*L is one
    int4 *tiles_s = reinterpret_cast<int4 *>(perm_s + T + ((4 - ((2 * T) & 3)) & 3));
    const int32_t *idx = STAGED ? idx_s : idx_g;

    if (STAGED)
        for (int t = threadIdx.x; t < T; t += blockDim.x) idx_s[t] = __ldg(idx_g + t);
    for (int i = threadIdx.x; i < kPlanWarps * L; i += blockDim.x) hist[i] = 0;
    if (threadIdx.x == 0) s_bad = 0;
    __syncthreads();

    const int per = ((T + kPlanWarps - 1) / kPlanWarps + 31) / 32 * 32;
    const int t_begin = min(T, warp * per), t_end = min(T, t_begin + per);
    int *my_hist = hist + warp * L;

    int n_inact = 0, bad = 0;
    for (int t0 = t_begin; t0 < t_end; t0 += 32) {  // warp-uniform
        const int t = t0 + lane;
        const bool live = t < t_end;
        int id = -1;
        if (live) {
            const int v = STAGED ? idx[t] : __ldg(idx + t);
            if (v >= 0 && v < L) id = v;
            else if (v != -1) bad++;
        }
        const unsigned peers = __match_any_sync(0xffffffffu, live ? id : -2);
        const unsigned inact = __ballot_sync(0xffffffffu, live && id < 0);
        if (live && id >= 0 && lane == __ffs(peers) - 1) my_hist[id] += __popc(peers);
        n_inact += __popc(inact);
    }
    if (bad) atomicAdd(&s_bad, bad);
    if (lane == 0) s_inact[warp] = n_inact;
    __syncthreads();

    // Thread l: adapter l's total and every warp's first slot for it.
    const int l = threadIdx.x;
    int cnt = 0;
    if (l < L) {
        for (int w = 0; w < kPlanWarps; ++w) {
            const int h = hist[w * L + l];
            hist[w * L + l] = cnt;
            cnt += h;
        }
    }
    int n_active;
    const int off = block_exclusive_scan(l < L ? cnt : 0, ws, &n_active);
    if (l < L) {
        p.count[l] = cnt;
        p.offset[l] = off;
        for (int w = 0; w < kPlanWarps; ++w) hist[w * L + l] += off;
    }
    if (threadIdx.x == 0) {
        p.offset[L] = n_active;
        int acc = n_active;
        for (int w = 0; w < kPlanWarps; ++w) {
            const int c = s_inact[w];
            s_inact[w] = acc;
            acc += c;
        }
    }
    __syncthreads();

    int ibase = s_inact[warp];
    const unsigned lt = (1u << lane) - 1u;
    for (int t0 = t_begin; t0 < t_end; t0 += 32) {
        const int t = t0 + lane;
        const bool live = t < t_end;
        int id = -1;
        if (live) {
            const int v = STAGED ? idx[t] : __ldg(idx + t);
            if (v >= 0 && v < L) id = v;
        }
        const unsigned peers = __match_any_sync(0xffffffffu, live ? id : -2);
        const unsigned inact = __ballot_sync(0xffffffffu, live && id < 0);
        if (live) {
            const int pos = id >= 0 ? my_hist[id] + __popc(peers & lt) : ibase + __popc(inact & lt);
            p.perm[pos] = t;
            if (STAGED) perm_s[pos] = t;
        }
        __syncwarp();
        if (live && id >= 0 && lane == __ffs(peers) - 1) my_hist[id] += __popc(peers);
        ibase += __popc(inact);
        __syncwarp();
    }

    // Groups: the adapters with at least one token, in ascending id.
    int G;
    const int has = (l < L && cnt > 0) ? 1 : 0;
    const int gi = block_exclusive_scan(has, ws, &G);
    if (has) {
        p.group_lora[gi] = l;
        p.group_start[gi] = off;
        p.group_count[gi] = cnt;
    }
    __syncthreads();
    if (STAGED) emit_tiles(p, T, n_active, G, ws, perm_s, tiles_s);
    else emit_tiles(p, T, n_active, G, ws);
    write_header(p, T, L, 1, n_active, G, s_bad, 0);
}

// ---------------------------------------------------------------- SGMV
struct SegClass {
    int st, ln, lora;     // lora after the bad-id rule
    bool active;          // valid, non-empty, adapter >= 0
    int err;              // LORA_PLANERR_* bits raised by this segment
    bool bad;             // counted as a bad id
};

// Classifies the segment of this thread within one 1024-segment chunk.
// carry_end: largest end of an in-range non-empty segment in earlier chunks.
__device__ SegClass classify(const int32_t *ss, const int32_t *sl, const int32_t *slo, int i,
                             int S, int T, int L, int carry_end, int *ws, int *chunk_max_end) {
    SegClass c{0, 0, -1, false, 0, false};
    bool nonempty = false;
    if (i < S) {
        c.st = __ldg(ss + i);
        c.ln = __ldg(sl + i);
        c.lora = __ldg(slo + i);
        const bool inrange = c.st >= 0 && c.ln >= 0 && (long long)c.st + c.ln <= T;
        if (!inrange) c.err |= LORA_PLANERR_SEG_RANGE;
        nonempty = inrange && c.ln > 0;
    }
    const int prev = max(carry_end, block_exclusive_max(nonempty ? c.st + c.ln : INT_MIN, ws,
                                                        chunk_max_end));
    if (nonempty) {
        if (c.st < prev) {
            c.err |= LORA_PLANERR_SEG_ORDER;
        } else {
            if (!(c.lora >= -1 && c.lora < L)) {
                c.bad = true;
                c.lora = -1;
            }
            c.active = c.lora >= 0;
        }
    }
    return c;
}

// Two passes over the segment table in chunks of 1024: pass 1 counts the
// active tokens (inactive tokens are placed after them), pass 2 writes perm,
// groups and per-adapter counts.  Active segments are disjoint and ascending
// by construction, so the tokens between two active segments are exactly
// the inactive ones, and inactive token t placed after active segment i-1
// has rank t - pos_i among the inactive tokens.
__global__ void __launch_bounds__(kPlanThreads, 1)
group_segments_kernel(const int32_t *__restrict__ ss, const int32_t *__restrict__ sl,
                      const int32_t *__restrict__ slo, int S, int T, int L, PlanPtrs p) {
    __shared__ int ws[40];
    __shared__ int sh_lora[kPlanThreads], sh_end[kPlanThreads];
    __shared__ int s_err, s_bad;
    const int lane = threadIdx.x & 31;
    grid_dep_wait();
    grid_dep_launch();  // dependents read the plan only after their own wait

    for (int l = threadIdx.x; l < L; l += blockDim.x) p.count[l] = 0;
    if (threadIdx.x == 0) {
        s_err = 0;
        s_bad = 0;
    }
    __syncthreads();

    // pass 1: number of active tokens
    int carry_end = 0, n_active = 0;
    for (int base = 0; base < S; base += blockDim.x) {
        int cmax, tot;
        const SegClass c = classify(ss, sl, slo, base + threadIdx.x, S, T, L, carry_end, ws, &cmax);
        block_exclusive_scan(c.active ? c.ln : 0, ws, &tot);
        carry_end = max(carry_end, cmax);
        n_active += tot;
    }

    // pass 2
    carry_end = 0;
    int carry_pos = 0, carry_groups = 0;
    int last_lora = -2, last_end = 0;  // previous active segment (lora -2 = none yet)
    for (int base = 0; base < S; base += blockDim.x) {
        const int i = base + threadIdx.x;
        int cmax, tot, ng, last_idx;
        const SegClass c = classify(ss, sl, slo, i, S, T, L, carry_end, ws, &cmax);
        if (c.err) atomicOr(&s_err, c.err);
        if (c.bad) atomicAdd(&s_bad, 1);
        const int pos = carry_pos + block_exclusive_scan(c.active ? c.ln : 0, ws, &tot);
        const int prev_local = block_exclusive_max(c.active ? (int)threadIdx.x : -1, ws, &last_idx);
        sh_lora[threadIdx.x] = c.lora;
        sh_end[threadIdx.x] = c.active ? c.st + c.ln : 0;
        __syncthreads();
        const int prev_lora = prev_local >= 0 ? sh_lora[prev_local] : last_lora;
        const int prev_end = prev_local >= 0 ? sh_end[prev_local] : last_end;
        const bool newgroup = c.active && prev_lora != c.lora;
        const int gid = carry_groups + block_exclusive_scan(newgroup ? 1 : 0, ws, &ng);
        if (newgroup) {
            p.group_lora[gid] = c.lora;
            p.group_start[gid] = pos;
        }
        if (c.active) atomicAdd(p.count + c.lora, c.ln);

        // Warp-cooperative placement: each warp walks its 32 segments.
        for (int j = 0; j < 32; ++j) {
            const bool a = __shfl_sync(0xffffffffu, c.active, j);
            if (!a) continue;
            const int st = __shfl_sync(0xffffffffu, c.st, j);
            const int ln = __shfl_sync(0xffffffffu, c.ln, j);
            const int ps = __shfl_sync(0xffffffffu, pos, j);
            const int gb = __shfl_sync(0xffffffffu, prev_end, j);
            for (int k = lane; k < ln; k += 32) p.perm[ps + k] = st + k;
            for (int t = gb + lane; t < st; t += 32) p.perm[n_active + t - ps] = t;
        }

        if (last_idx >= 0) {
            last_lora = sh_lora[last_idx];
            last_end = sh_end[last_idx];
        }
        carry_end = max(carry_end, cmax);
        carry_pos += tot;
        carry_groups += ng;
        __syncthreads();
    }
    // inactive tail after the last active segment: rank t - n_active
    for (int t = last_end + threadIdx.x; t < T; t += blockDim.x) p.perm[t] = t;
    const int G = carry_groups;
    __syncthreads();
    for (int g = threadIdx.x; g < G; g += blockDim.x)
        p.group_count[g] = (g + 1 < G ? p.group_start[g + 1] : n_active) - p.group_start[g];
    __syncthreads();
    // per-adapter offsets (L <= LORA_MAX_ADAPTERS = blockDim.x)
    int total;
    const int l = threadIdx.x;
    const int cnt = l < L ? __ldcg(p.count + l) : 0;  // written by atomics
    const int off = block_exclusive_scan(cnt, ws, &total);
    if (l < L) p.offset[l] = off;
    if (threadIdx.x == 0) p.offset[L] = total;
    emit_tiles(p, T, n_active, G, ws);
    write_header(p, T, L, 2, n_active, G, s_bad, s_err);
}

}  // namespace

static_assert(LORA_MAX_ADAPTERS <= kPlanThreads, "one thread per adapter");

// Small batches (decode) use 8 warps: fewer threads make the block-wide
// scans and barriers of this latency-bound kernel cheaper; above 512 tokens
// 16 warps (T = 1024: 4.8 -> 4.4 us; 32 warps measured slower).
constexpr int kSmallWarps = 8;
constexpr int kMidWarps = 16;
constexpr int kMidMinT = 513;
constexpr int kSmallMaxT = 8192;

// Shared memory of the staged variant with nw warps: histogram, idx, perm,
// tile records.
size_t staged_smem(int T, int L, int nw) {
    const size_t tiles = (size_t)(T / kTile + std::min(L, T) + 2);
    return sizeof(int) * ((size_t)nw * L + 2 * (size_t)T + 4) + 16 * tiles;
}

cudaError_t configure_plan_kernels() {
    cudaError_t e = cudaFuncSetAttribute(group_tokens_kernel<kPlanWarps, false>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)(sizeof(int) * kPlanWarps * LORA_MAX_ADAPTERS));
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(group_tokens_kernel<kMidWarps, true>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)staged_smem(kSmallMaxT, kSmallWarps * 32, kMidWarps));
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(group_tokens_kernel<kSmallWarps, true>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)staged_smem(kSmallMaxT, kSmallWarps * 32, kSmallWarps));
}

cudaError_t launch_group_tokens(const int32_t *idx, int T, int L, const PlanPtrs &p,
                                cudaStream_t stream) {
    if (T >= kMidMinT && T <= kSmallMaxT && L <= kSmallWarps * 32) {
        group_tokens_kernel<kMidWarps, true>
            <<<1, kMidWarps * 32, staged_smem(T, L, kMidWarps), stream>>>(idx, T, L, p);
    } else if (T <= kSmallMaxT && L <= kSmallWarps * 32) {
        group_tokens_kernel<kSmallWarps, true>
            <<<1, kSmallWarps * 32, staged_smem(T, L, kSmallWarps), stream>>>(idx, T, L, p);
    } else {
        const size_t smem = sizeof(int) * kPlanWarps * (size_t)L;
        group_tokens_kernel<kPlanWarps, false><<<1, kPlanThreads, smem, stream>>>(idx, T, L, p);
    }
    return cudaGetLastError();
}

cudaError_t launch_group_segments(const int32_t *ss, const int32_t *sl, const int32_t *slo,
                                  int S, int T, int L, const PlanPtrs &p, cudaStream_t stream) {
    group_segments_kernel<<<1, kPlanThreads, 0, stream>>>(ss, sl, slo, S, T, L, p);
    return cudaGetLastError();
}

}  // namespace lora
