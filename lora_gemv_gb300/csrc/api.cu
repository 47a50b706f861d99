// C ABI layer: argument validation, per-device set-up and dispatch.
// Declarations and the meaning of every argument: include/lora_gemv.h.
#include <stdarg.h>
#include <stdio.h>

#include <algorithm>
#include <mutex>
#include <unordered_set>

#include "kernels.h"

namespace {

thread_local char g_detail[512] = "";

lora_status_t fail(lora_status_t s, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_detail, sizeof(g_detail), fmt, ap);
    va_end(ap);
    return s;
}

lora_status_t cuda_fail(cudaError_t e, const char *what) {
    return fail(LORA_ERR_CUDA, "%s: %s (%d)", what, cudaGetErrorString(e), (int)e);
}

constexpr int kMaxDevices = 64;
struct DevState {
    std::once_flag once;
    cudaError_t err = cudaSuccess;
    lora::DeviceInfo info{};
};
DevState g_dev[kMaxDevices];

cudaError_t init_device(int dev, lora::DeviceInfo *info) {
    cudaError_t e = cudaDeviceGetAttribute(&info->sm_count, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    if ((e = lora::configure_plan_kernels()) != cudaSuccess) return e;
    if ((e = lora::configure_shrink_kernels(info)) != cudaSuccess) return e;
    if ((e = lora::configure_expand_kernels()) != cudaSuccess) return e;
    if ((e = lora::configure_bgmv_kernels(*info)) != cudaSuccess) return e;
    return lora::configure_fused_kernels(*info);
}

// Per-device kernel attributes are set once, on the first call on that device.
lora_status_t device_info(const lora::DeviceInfo **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) return fail(LORA_ERR_UNSUPPORTED, "device %d", dev);
    DevState &d = g_dev[dev];
    std::call_once(d.once, [&] { d.err = init_device(dev, &d.info); });
    if (d.err != cudaSuccess) return cuda_fail(d.err, "device set-up");
    *out = &d.info;
    return LORA_OK;
}

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

lora_status_t check_plan(const void *plan, size_t plan_bytes, int32_t T, int32_t L,
                         lora_plan_layout_t *lay) {
    lora_status_t s = lora_plan_layout(T, L, lay);
    if (s != LORA_OK) return s;
    if (plan == nullptr) return fail(LORA_ERR_INVALID_ARG, "plan is NULL");
    if (!aligned(plan, 16)) return fail(LORA_ERR_WORKSPACE, "plan is not 16-byte aligned");
    if (plan_bytes < (size_t)lay->bytes)
        return fail(LORA_ERR_WORKSPACE, "plan buffer has %zu bytes, needs %lld", plan_bytes,
                    (long long)lay->bytes);
    return LORA_OK;
}

lora::PlanPtrs plan_ptrs(void *plan, const lora_plan_layout_t &lay) {
    char *b = static_cast<char *>(plan);
    lora::PlanPtrs p;
    p.hdr = reinterpret_cast<int32_t *>(b + lay.header);
    p.count = reinterpret_cast<int32_t *>(b + lay.count);
    p.offset = reinterpret_cast<int32_t *>(b + lay.offset);
    p.perm = reinterpret_cast<int32_t *>(b + lay.perm);
    p.group_lora = reinterpret_cast<int32_t *>(b + lay.group_lora);
    p.group_start = reinterpret_cast<int32_t *>(b + lay.group_start);
    p.group_count = reinterpret_cast<int32_t *>(b + lay.group_count);
    p.tiles = reinterpret_cast<int4 *>(b + lay.tiles);
    p.tile_rows = reinterpret_cast<int32_t *>(b + lay.tile_rows);
    return p;
}

bool valid_dtype(lora_dtype_t d) { return d == LORA_F16 || d == LORA_BF16; }

}  // namespace

extern "C" {

lora_status_t lora_plan_layout(int32_t T, int32_t L, lora_plan_layout_t *lay) {
    if (lay == nullptr) return fail(LORA_ERR_INVALID_ARG, "layout is NULL");
    if (T < 0) return fail(LORA_ERR_INVALID_ARG, "T = %d < 0", T);
    if (L < 1) return fail(LORA_ERR_INVALID_ARG, "L = %d < 1", L);
    if (T > LORA_MAX_TOKENS) return fail(LORA_ERR_UNSUPPORTED, "T = %d > %d", T, LORA_MAX_TOKENS);
    if (L > LORA_MAX_ADAPTERS)
        return fail(LORA_ERR_UNSUPPORTED, "L = %d > %d", L, LORA_MAX_ADAPTERS);
    int64_t off = 0;
    lay->header = off;
    off += LORA_HDR_WORDS * 4;
    lay->count = off;
    off += (int64_t)L * 4;
    lay->offset = off;
    off += (int64_t)(L + 1) * 4;
    lay->perm = off;
    off += (int64_t)T * 4;
    lay->group_lora = off;
    off += (int64_t)(T + 1) * 4;
    lay->group_start = off;
    off += (int64_t)(T + 1) * 4;
    lay->group_count = off;
    off += (int64_t)(T + 1) * 4;
    off = (off + 15) / 16 * 16;
    lay->tiles = off;
    lay->max_tiles = (int64_t)T + T / LORA_TILE_TOKENS + 2;
    off += lay->max_tiles * 16;
    lay->tile_rows = off;
    off += lay->max_tiles * LORA_TILE_TOKENS * 4;
    lay->bytes = off;
    return LORA_OK;
}

size_t lora_workspace_size(int32_t T, int32_t L) {
    lora_plan_layout_t lay;
    return lora_plan_layout(T, L, &lay) == LORA_OK ? (size_t)lay.bytes : 0;
}

}  // extern "C"

namespace {
// Plans grouped by this library from a segment table, by address.  A hint for
// the shrink's launch shape only (segment plans mostly hold tiles of
// consecutive token rows, which the TMA-staging variant copies in bulk);
// every variant checks each tile itself, so a stale entry costs speed, never
// correctness.
std::mutex g_kind_mu;
std::unordered_set<const void *> g_seg_plans;
void note_plan_kind(const void *plan, bool segments) {
    std::lock_guard<std::mutex> lk(g_kind_mu);
    if (segments) g_seg_plans.insert(plan);
    else g_seg_plans.erase(plan);
}
bool is_seg_plan(const void *plan) {
    std::lock_guard<std::mutex> lk(g_kind_mu);
    return g_seg_plans.count(plan) != 0;
}
}  // namespace

extern "C" {

lora_status_t lora_group_tokens(const int32_t *token_idx, int32_t T, int32_t L, void *plan,
                                size_t plan_bytes, lora_stream_t stream) {
    lora_plan_layout_t lay;
    lora_status_t s = check_plan(plan, plan_bytes, T, L, &lay);
    if (s != LORA_OK) return s;
    if (T > 0 && token_idx == nullptr) return fail(LORA_ERR_INVALID_ARG, "token_idx is NULL");
    if (!aligned(token_idx, 4)) return fail(LORA_ERR_INVALID_ARG, "token_idx misaligned");
    const lora::DeviceInfo *dev;
    if ((s = device_info(&dev)) != LORA_OK) return s;
    note_plan_kind(plan, false);
    cudaError_t e = lora::launch_group_tokens(token_idx, T, L, plan_ptrs(plan, lay),
                                              reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? LORA_OK : cuda_fail(e, "group_tokens launch");
}

lora_status_t lora_group_segments(const int32_t *seg_start, const int32_t *seg_len,
                                  const int32_t *seg_lora, int32_t num_segs, int32_t T, int32_t L,
                                  void *plan, size_t plan_bytes, lora_stream_t stream) {
    lora_plan_layout_t lay;
    lora_status_t s = check_plan(plan, plan_bytes, T, L, &lay);
    if (s != LORA_OK) return s;
    if (num_segs < 0) return fail(LORA_ERR_INVALID_ARG, "num_segs = %d < 0", num_segs);
    if (num_segs > 0 && (!seg_start || !seg_len || !seg_lora))
        return fail(LORA_ERR_INVALID_ARG, "segment table pointer is NULL");
    if (!aligned(seg_start, 4) || !aligned(seg_len, 4) || !aligned(seg_lora, 4))
        return fail(LORA_ERR_INVALID_ARG, "segment table misaligned");
    const lora::DeviceInfo *dev;
    if ((s = device_info(&dev)) != LORA_OK) return s;
    note_plan_kind(plan, true);
    cudaError_t e = lora::launch_group_segments(seg_start, seg_len, seg_lora, num_segs, T, L,
                                                plan_ptrs(plan, lay),
                                                reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? LORA_OK : cuda_fail(e, "group_segments launch");
}

}  // extern "C"

namespace lora {

// Reports a failure status with a message (the thread's lora_last_error_detail).
lora_status_t report(lora_status_t s, const char *msg) { return fail(s, "%s", msg); }

lora_status_t check_shrink(lora_dtype_t dtype, const void *x, int64_t ldx, int32_t T, int32_t H,
                           const void *A, int32_t L, int32_t R, int32_t num_slices,
                           const int32_t *ranks, const float *y, int64_t ldy, const void *plan) {
    if (!valid_dtype(dtype)) return fail(LORA_ERR_INVALID_ARG, "dtype %d", (int)dtype);
    if (T < 0 || H < 1 || L < 1) return fail(LORA_ERR_INVALID_ARG, "T=%d H=%d L=%d", T, H, L);
    if (R < 1 || R > LORA_MAX_RANK) return fail(LORA_ERR_INVALID_ARG, "R = %d", R);
    if (num_slices < 1 || num_slices > LORA_MAX_SLICES)
        return fail(LORA_ERR_INVALID_ARG, "num_slices = %d", num_slices);
    if (ldx < H) return fail(LORA_ERR_INVALID_ARG, "ldx %lld < H %d", (long long)ldx, H);
    if (ldy < (int64_t)num_slices * R)
        return fail(LORA_ERR_INVALID_ARG, "ldy %lld < num_slices*R", (long long)ldy);
    if (!A || !plan || (T > 0 && (!x || !y))) return fail(LORA_ERR_INVALID_ARG, "NULL pointer");
    if (!aligned(x, 2) || !aligned(A, 2) || !aligned(y, 4) || !aligned(ranks, 4))
        return fail(LORA_ERR_INVALID_ARG, "misaligned pointer");
    if (!aligned(plan, 16)) return fail(LORA_ERR_WORKSPACE, "plan is not 16-byte aligned");
    lora_plan_layout_t lay;
    return lora_plan_layout(T, L, &lay);
}

lora_status_t check_expand(lora_dtype_t dtype, const float *y, int64_t ldy, int32_t T,
                           int32_t num_slices, const void *const *B_slices,
                           const int32_t *slice_N, const int32_t *slice_offset,
                           int32_t y_slice_stride, int32_t L, int32_t R, const int32_t *ranks,
                           const void *out, int64_t ldo, const void *plan) {
    if (!valid_dtype(dtype)) return fail(LORA_ERR_INVALID_ARG, "dtype %d", (int)dtype);
    if (T < 0 || L < 1) return fail(LORA_ERR_INVALID_ARG, "T=%d L=%d", T, L);
    if (R < 1 || R > LORA_MAX_RANK) return fail(LORA_ERR_INVALID_ARG, "R = %d", R);
    if (num_slices < 1 || num_slices > LORA_MAX_SLICES)
        return fail(LORA_ERR_INVALID_ARG, "num_slices = %d", num_slices);
    if (!B_slices || !slice_N || !slice_offset)
        return fail(LORA_ERR_INVALID_ARG, "slice arrays are NULL");
    if (y_slice_stride < 0) return fail(LORA_ERR_INVALID_ARG, "y_slice_stride < 0");
    if ((int64_t)(num_slices - 1) * y_slice_stride + R > ldy)
        return fail(LORA_ERR_INVALID_ARG, "y columns of the last slice exceed ldy");
    if (!plan || (T > 0 && (!y || !out))) return fail(LORA_ERR_INVALID_ARG, "NULL pointer");
    if (!aligned(y, 4) || !aligned(out, 2) || !aligned(ranks, 4))
        return fail(LORA_ERR_INVALID_ARG, "misaligned pointer");
    if (!aligned(plan, 16)) return fail(LORA_ERR_WORKSPACE, "plan is not 16-byte aligned");
    int order[LORA_MAX_SLICES];
    for (int s = 0; s < num_slices; ++s) {
        if (slice_N[s] < 0 || slice_offset[s] < 0)
            return fail(LORA_ERR_INVALID_ARG, "slice %d: N=%d offset=%d", s, slice_N[s],
                        slice_offset[s]);
        if ((int64_t)slice_offset[s] + slice_N[s] > ldo)
            return fail(LORA_ERR_INVALID_ARG, "slice %d ends past ldo", s);
        if (slice_N[s] > 0 && (B_slices[s] == nullptr || !aligned(B_slices[s], 2)))
            return fail(LORA_ERR_INVALID_ARG, "slice %d weights NULL or misaligned", s);
        order[s] = s;
    }
    std::sort(order, order + num_slices,
              [&](int i, int j) { return slice_offset[i] < slice_offset[j]; });
    for (int k = 0; k + 1 < num_slices; ++k) {
        const int i = order[k], j = order[k + 1];
        if (slice_N[i] > 0 && slice_N[j] > 0 && slice_offset[i] + slice_N[i] > slice_offset[j])
            return fail(LORA_ERR_INVALID_ARG, "slices %d and %d overlap", i, j);
    }
    lora_plan_layout_t lay;
    return lora_plan_layout(T, L, &lay);
}

}  // namespace lora

using lora::check_expand;
using lora::check_shrink;

extern "C" {

lora_status_t lora_shrink(lora_dtype_t dtype, const void *x, int64_t ldx, int32_t T, int32_t H,
                          const void *A, int32_t L, int32_t R, int32_t num_slices,
                          const int32_t *ranks, float *y, int64_t ldy, const void *plan,
                          float scale, int add_inputs, lora_stream_t stream) {
    {
        lora_status_t st = check_shrink(dtype, x, ldx, T, H, A, L, R, num_slices, ranks, y, ldy, plan);
        if (st != LORA_OK) return st;
    }
    lora_plan_layout_t lay;
    lora_status_t s = lora_plan_layout(T, L, &lay);
    if (s != LORA_OK) return s;
    if (T == 0) return LORA_OK;
    const lora::DeviceInfo *dev;
    if ((s = device_info(&dev)) != LORA_OK) return s;
    lora::PlanPtrs p = plan_ptrs(const_cast<void *>(plan), lay);
    lora::ShrinkArgs a{};
    a.x = x;
    a.ldx = ldx;
    a.T = T;
    a.H = H;
    a.A = A;
    a.L = L;
    a.R = R;
    a.S = num_slices;
    a.ranks = ranks;
    a.y = y;
    a.ldy = ldy;
    a.scale = scale;
    a.add = add_inputs ? 1 : 0;
    a.hdr = p.hdr;
    a.perm = p.perm;
    a.tiles = p.tiles;
    a.tile_rows = p.tile_rows;
    a.max_tiles = (int)lay.max_tiles;
    a.seg_plan = is_seg_plan(plan) ? 1 : 0;
    cudaError_t e = lora::launch_shrink(dtype, a, *dev, reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? LORA_OK : cuda_fail(e, "shrink launch");
}

lora_status_t lora_expand_slice(lora_dtype_t dtype, const float *y, int64_t ldy, int32_t T,
                                int32_t num_slices, const void *const *B_slices,
                                const int32_t *slice_N, const int32_t *slice_offset,
                                int32_t y_slice_stride, int32_t L, int32_t R,
                                const int32_t *ranks, void *out, int64_t ldo, const void *plan,
                                float scale, int add_inputs, lora_stream_t stream) {
    {
        lora_status_t st = check_expand(dtype, y, ldy, T, num_slices, B_slices, slice_N,
                                        slice_offset, y_slice_stride, L, R, ranks, out, ldo, plan);
        if (st != LORA_OK) return st;
    }
    lora_plan_layout_t lay;
    lora_status_t s = lora_plan_layout(T, L, &lay);
    if (s != LORA_OK) return s;
    if (T == 0) return LORA_OK;
    const lora::DeviceInfo *dev;
    if ((s = device_info(&dev)) != LORA_OK) return s;
    lora::PlanPtrs p = plan_ptrs(const_cast<void *>(plan), lay);
    lora::ExpandArgs a{};
    a.y = y;
    a.ldy = ldy;
    a.T = T;
    a.out = out;
    a.ldo = ldo;
    a.L = L;
    a.R = R;
    a.ranks = ranks;
    a.y_slice_stride = y_slice_stride;
    a.scale = scale;
    a.add = add_inputs ? 1 : 0;
    a.num_slices = num_slices;
    for (int k = 0; k < num_slices; ++k) {
        a.B[k] = B_slices[k];
        a.N[k] = slice_N[k];
        a.off[k] = slice_offset[k];
    }
    a.hdr = p.hdr;
    a.perm = p.perm;
    a.tiles = p.tiles;
    a.tile_rows = p.tile_rows;
    a.max_tiles = (int)lay.max_tiles;
    a.seg_plan = is_seg_plan(plan) ? 1 : 0;
    cudaError_t e = lora::launch_expand(dtype, a, *dev, reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? LORA_OK : cuda_fail(e, "expand launch");
}

lora_status_t lora_expand(lora_dtype_t dtype, const float *y, int64_t ldy, int32_t T,
                          const void *B, int32_t L, int32_t N, int32_t R, const int32_t *ranks,
                          void *out, int64_t ldo, const void *plan, float scale, int add_inputs,
                          lora_stream_t stream) {
    const void *Bs[1] = {B};
    const int32_t Ns[1] = {N};
    const int32_t offs[1] = {0};
    return lora_expand_slice(dtype, y, ldy, T, 1, Bs, Ns, offs, 0, L, R, ranks, out, ldo, plan,
                             scale, add_inputs, stream);
}

lora_status_t lora_shrink_expand_slice(lora_dtype_t dtype, const void *x, int64_t ldx, int32_t T,
                                       int32_t H, const void *A, int32_t L, int32_t R,
                                       const int32_t *ranks, float *y, int64_t ldy,
                                       int32_t num_slices, const void *const *B_slices,
                                       const int32_t *slice_N, const int32_t *slice_offset,
                                       void *out, int64_t ldo, const void *plan,
                                       float scale_shrink, float scale_expand, int add_inputs,
                                       lora_stream_t stream) {
    lora_status_t st = check_shrink(dtype, x, ldx, T, H, A, L, R, num_slices, ranks, y, ldy, plan);
    if (st != LORA_OK) return st;
    st = check_expand(dtype, y, ldy, T, num_slices, B_slices, slice_N, slice_offset, R, L, R, ranks,
                      out, ldo, plan);
    if (st != LORA_OK) return st;
    if (T == 0) return LORA_OK;
    const lora::DeviceInfo *dev;
    if ((st = device_info(&dev)) != LORA_OK) return st;
    lora_plan_layout_t lay;
    lora_plan_layout(T, L, &lay);
    lora::PlanPtrs p = plan_ptrs(const_cast<void *>(plan), lay);
    cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    lora::ShrinkArgs sa{};
    sa.x = x;
    sa.ldx = ldx;
    sa.T = T;
    sa.H = H;
    sa.A = A;
    sa.L = L;
    sa.R = R;
    sa.S = num_slices;
    sa.ranks = ranks;
    sa.y = y;
    sa.ldy = ldy;
    sa.scale = scale_shrink;
    sa.add = 0;
    sa.hdr = p.hdr;
    sa.perm = p.perm;
    sa.tiles = p.tiles;
    sa.tile_rows = p.tile_rows;
    sa.max_tiles = (int)lay.max_tiles;
    sa.seg_plan = is_seg_plan(plan) ? 1 : 0;
    lora::ExpandArgs ea{};
    ea.y = y;
    ea.ldy = ldy;
    ea.T = T;
    ea.out = out;
    ea.ldo = ldo;
    ea.L = L;
    ea.R = R;
    ea.ranks = ranks;
    ea.y_slice_stride = R;
    ea.scale = scale_expand;
    ea.add = add_inputs ? 1 : 0;
    ea.num_slices = num_slices;
    for (int k = 0; k < num_slices; ++k) {
        ea.B[k] = B_slices[k];
        ea.N[k] = slice_N[k];
        ea.off[k] = slice_offset[k];
    }
    ea.hdr = p.hdr;
    ea.perm = p.perm;
    ea.tiles = p.tiles;
    ea.tile_rows = p.tile_rows;
    ea.max_tiles = (int)lay.max_tiles;
    ea.seg_plan = is_seg_plan(plan) ? 1 : 0;
    ea.early = 1;
    // The shrink waits for the caller's previous kernels, then lets the
    // expand launch early; the expand reads plan, out and B (none written by
    // the shrink) before its own wait and y after it.
    cudaError_t e = lora::launch_shrink(dtype, sa, *dev, cs, true);
    if (e == cudaSuccess) e = lora::launch_expand(dtype, ea, *dev, cs, true);
    return e == cudaSuccess ? LORA_OK : cuda_fail(e, "shrink_expand_slice launch");
}

lora_status_t lora_get_error(const void *plan, int32_t *bad_ids, int32_t *err_flags,
                             lora_stream_t stream) {
    if (plan == nullptr) return fail(LORA_ERR_INVALID_ARG, "plan is NULL");
    int32_t hdr[LORA_HDR_WORDS];
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = cudaMemcpyAsync(hdr, plan, sizeof(hdr), cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return cuda_fail(e, "reading the plan header");
    if (bad_ids) *bad_ids = hdr[LORA_HDR_BAD_IDS];
    if (err_flags) *err_flags = hdr[LORA_HDR_ERR];
    return LORA_OK;
}

const char *lora_status_string(lora_status_t status) {
    switch (status) {
    case LORA_OK: return "ok";
    case LORA_ERR_INVALID_ARG: return "invalid argument";
    case LORA_ERR_UNSUPPORTED: return "unsupported size or configuration";
    case LORA_ERR_WORKSPACE: return "plan buffer too small or misaligned";
    case LORA_ERR_CUDA: return "CUDA runtime error";
    }
    return "unknown status";
}

const char *lora_last_error_detail(void) { return g_detail; }

int32_t lora_version(void) { return 100; }

}  // extern "C"

// ------------------------------------------------------------------ plan-free BGMV

namespace {

lora_status_t check_bgmv_shrink(lora_dtype_t dtype, const int32_t *token_idx, const void *x,
                                int64_t ldx, int32_t T, int32_t H, const void *A, int32_t L,
                                int32_t R, int32_t num_slices, const int32_t *ranks,
                                const float *y, int64_t ldy) {
    if (!valid_dtype(dtype)) return fail(LORA_ERR_INVALID_ARG, "dtype %d", (int)dtype);
    if (T < 0 || H < 1 || L < 1) return fail(LORA_ERR_INVALID_ARG, "T=%d H=%d L=%d", T, H, L);
    if (R < 1 || R > LORA_MAX_RANK) return fail(LORA_ERR_INVALID_ARG, "R = %d", R);
    if (num_slices < 1 || num_slices > LORA_MAX_SLICES)
        return fail(LORA_ERR_INVALID_ARG, "num_slices = %d", num_slices);
    if (ldx < H) return fail(LORA_ERR_INVALID_ARG, "ldx %lld < H %d", (long long)ldx, H);
    if (ldy < (int64_t)num_slices * R)
        return fail(LORA_ERR_INVALID_ARG, "ldy %lld < num_slices*R", (long long)ldy);
    if (!A || (T > 0 && (!x || !y))) return fail(LORA_ERR_INVALID_ARG, "NULL pointer");
    if (!aligned(token_idx, 4) || !aligned(y, 4) || !aligned(ranks, 4))
        return fail(LORA_ERR_INVALID_ARG, "misaligned pointer");
    if (T > LORA_BGMV_MAX_TOKENS)
        return fail(LORA_ERR_UNSUPPORTED, "T = %d > %d", T, LORA_BGMV_MAX_TOKENS);
    if (L > LORA_BGMV_MAX_ADAPTERS)
        return fail(LORA_ERR_UNSUPPORTED, "L = %d > %d (use the grouped operators)", L,
                    LORA_BGMV_MAX_ADAPTERS);
    return LORA_OK;
}

lora_status_t check_bgmv_expand(lora_dtype_t dtype, const int32_t *token_idx, const float *y,
                                int64_t ldy, int32_t T, int32_t num_slices,
                                const void *const *B_slices, const int32_t *slice_N,
                                const int32_t *slice_offset, int32_t y_slice_stride, int32_t L,
                                int32_t R, const int32_t *ranks, const void *out, int64_t ldo) {
    if (T > LORA_BGMV_MAX_TOKENS)
        return fail(LORA_ERR_UNSUPPORTED, "T = %d > %d", T, LORA_BGMV_MAX_TOKENS);
    if (L > LORA_BGMV_MAX_ADAPTERS)
        return fail(LORA_ERR_UNSUPPORTED, "L = %d > %d (use the grouped operators)", L,
                    LORA_BGMV_MAX_ADAPTERS);
    if (!aligned(token_idx, 4)) return fail(LORA_ERR_INVALID_ARG, "token_idx misaligned");
    // the grouped operator's checks, with a stand-in for its plan argument
    static const int4 no_plan = {0, 0, 0, 0};
    return check_expand(dtype, y, ldy, T, num_slices, B_slices, slice_N, slice_offset,
                        y_slice_stride, L, R, ranks, out, ldo, &no_plan);
}

lora::BgmvShrinkArgs bgmv_shrink_args(const int32_t *token_idx, const void *x, int64_t ldx,
                                      int32_t T, int32_t H, const void *A, int32_t L, int32_t R,
                                      int32_t num_slices, const int32_t *ranks, float *y,
                                      int64_t ldy, float scale, int add_inputs,
                                      int32_t *status) {
    lora::BgmvShrinkArgs a{};
    a.x = x;
    a.ldx = ldx;
    a.T = T;
    a.H = H;
    a.A = A;
    a.L = L;
    a.R = R;
    a.S = num_slices;
    a.idx = token_idx;
    a.ranks = ranks;
    a.y = y;
    a.ldy = ldy;
    a.scale = scale;
    a.add = add_inputs ? 1 : 0;
    a.status = status;
    return a;
}

lora::BgmvExpandArgs bgmv_expand_args(const int32_t *token_idx, const float *y, int64_t ldy,
                                      int32_t T, int32_t num_slices,
                                      const void *const *B_slices, const int32_t *slice_N,
                                      const int32_t *slice_offset, int32_t y_slice_stride,
                                      int32_t L, int32_t R, const int32_t *ranks, void *out,
                                      int64_t ldo, float scale, int add_inputs,
                                      int32_t *status) {
    lora::BgmvExpandArgs a{};
    a.y = y;
    a.ldy = ldy;
    a.T = T;
    a.idx = token_idx;
    a.ranks = ranks;
    a.L = L;
    a.R = R;
    a.y_slice_stride = y_slice_stride;
    a.scale = scale;
    a.add = add_inputs ? 1 : 0;
    a.num_slices = num_slices;
    for (int k = 0; k < num_slices; ++k) {
        a.B[k] = B_slices[k];
        a.N[k] = slice_N[k];
        a.off[k] = slice_offset[k];
    }
    a.out = out;
    a.ldo = ldo;
    a.status = status;
    return a;
}

}  // namespace

extern "C" {

lora_status_t lora_bgmv_shrink(lora_dtype_t dtype, const int32_t *token_idx, const void *x,
                               int64_t ldx, int32_t T, int32_t H, const void *A, int32_t L,
                               int32_t R, int32_t num_slices, const int32_t *ranks, float *y,
                               int64_t ldy, float scale, int add_inputs, int32_t *status,
                               lora_stream_t stream) {
    lora_status_t st = check_bgmv_shrink(dtype, token_idx, x, ldx, T, H, A, L, R, num_slices,
                                         ranks, y, ldy);
    if (st != LORA_OK) return st;
    const lora::BgmvShrinkArgs a = bgmv_shrink_args(token_idx, x, ldx, T, H, A, L, R, num_slices,
                                                    ranks, y, ldy, scale, add_inputs, status);
    if (const char *why = lora::bgmv_shrink_supported(a)) return fail(LORA_ERR_UNSUPPORTED, "%s", why);
    if (T == 0) return LORA_OK;
    const lora::DeviceInfo *dev;
    if ((st = device_info(&dev)) != LORA_OK) return st;
    // programmatic launch: only the launch overlaps the previous kernel's
    // tail; every read waits for it
    cudaError_t e = lora::launch_bgmv_shrink(dtype, a, *dev, reinterpret_cast<cudaStream_t>(stream), true);
    return e == cudaSuccess ? LORA_OK : cuda_fail(e, "bgmv shrink launch");
}

lora_status_t lora_bgmv_expand_slice(lora_dtype_t dtype, const int32_t *token_idx, const float *y,
                                     int64_t ldy, int32_t T, int32_t num_slices,
                                     const void *const *B_slices, const int32_t *slice_N,
                                     const int32_t *slice_offset, int32_t y_slice_stride,
                                     int32_t L, int32_t R, const int32_t *ranks, void *out,
                                     int64_t ldo, float scale, int add_inputs, int32_t *status,
                                     lora_stream_t stream) {
    lora_status_t st = check_bgmv_expand(dtype, token_idx, y, ldy, T, num_slices, B_slices,
                                         slice_N, slice_offset, y_slice_stride, L, R, ranks, out,
                                         ldo);
    if (st != LORA_OK) return st;
    const lora::BgmvExpandArgs a =
        bgmv_expand_args(token_idx, y, ldy, T, num_slices, B_slices, slice_N, slice_offset,
                         y_slice_stride, L, R, ranks, out, ldo, scale, add_inputs, status);
    if (const char *why = lora::bgmv_expand_supported(a)) return fail(LORA_ERR_UNSUPPORTED, "%s", why);
    if (T == 0) return LORA_OK;
    const lora::DeviceInfo *dev;
    if ((st = device_info(&dev)) != LORA_OK) return st;
    // programmatic launch with early = 0: only the launch overlaps the
    // previous kernel's tail; every read waits for it
    cudaError_t e = lora::launch_bgmv_expand(dtype, a, *dev, reinterpret_cast<cudaStream_t>(stream), true);
    return e == cudaSuccess ? LORA_OK : cuda_fail(e, "bgmv expand launch");
}

lora_status_t lora_bgmv_shrink_expand_slice(
    lora_dtype_t dtype, const int32_t *token_idx, const void *x, int64_t ldx, int32_t T, int32_t H,
    const void *A, int32_t L, int32_t R, const int32_t *ranks, float *y, int64_t ldy,
    int32_t num_slices, const void *const *B_slices, const int32_t *slice_N,
    const int32_t *slice_offset, void *out, int64_t ldo, float scale_shrink, float scale_expand,
    int add_inputs, int32_t *status, lora_stream_t stream) {
    lora_status_t st = check_bgmv_shrink(dtype, token_idx, x, ldx, T, H, A, L, R, num_slices,
                                         ranks, y, ldy);
    if (st != LORA_OK) return st;
    st = check_bgmv_expand(dtype, token_idx, y, ldy, T, num_slices, B_slices, slice_N,
                           slice_offset, R, L, R, ranks, out, ldo);
    if (st != LORA_OK) return st;
    const lora::BgmvShrinkArgs sa = bgmv_shrink_args(token_idx, x, ldx, T, H, A, L, R, num_slices,
                                                     ranks, y, ldy, scale_shrink, 0, status);
    lora::BgmvExpandArgs ea =
        bgmv_expand_args(token_idx, y, ldy, T, num_slices, B_slices, slice_N, slice_offset, R, L,
                         R, ranks, out, ldo, scale_expand, add_inputs, status);
    ea.early = 1;  // the shrink writes only y
    if (const char *why = lora::bgmv_shrink_supported(sa)) return fail(LORA_ERR_UNSUPPORTED, "%s", why);
    if (const char *why = lora::bgmv_expand_supported(ea)) return fail(LORA_ERR_UNSUPPORTED, "%s", why);
    if (T == 0) return LORA_OK;
    const lora::DeviceInfo *dev;
    if ((st = device_info(&dev)) != LORA_OK) return st;
    cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    // The expand is a programmatic dependent of the shrink: it stages out and
    // B while the shrink runs and reads y after the shrink grid completes.
    cudaError_t e = lora::launch_bgmv_shrink(dtype, sa, *dev, cs, true);
    if (e == cudaSuccess) e = lora::launch_bgmv_expand(dtype, ea, *dev, cs, true);
    return e == cudaSuccess ? LORA_OK : cuda_fail(e, "bgmv shrink_expand_slice launch");
}

lora_status_t lora_bgmv_fused_shrink_expand_slice(
    lora_dtype_t dtype, const int32_t *token_idx, const void *x, int64_t ldx, int32_t T, int32_t H,
    const void *A, int32_t L, int32_t R, const int32_t *ranks, float *y, int64_t ldy,
    int32_t num_slices, const void *const *B_slices, const int32_t *slice_N,
    const int32_t *slice_offset, void *out, int64_t ldo, float scale_shrink, float scale_expand,
    int add_inputs, lora_stream_t stream) {
    lora_status_t st = check_bgmv_shrink(dtype, token_idx, x, ldx, T, H, A, L, R, num_slices,
                                         ranks, y, ldy);
    if (st != LORA_OK) return st;
    st = check_bgmv_expand(dtype, token_idx, y, ldy, T, num_slices, B_slices, slice_N,
                           slice_offset, R, L, R, ranks, out, ldo);
    if (st != LORA_OK) return st;
    const lora::BgmvShrinkArgs sa = bgmv_shrink_args(token_idx, x, ldx, T, H, A, L, R, num_slices,
                                                     ranks, y, ldy, scale_shrink, 0, nullptr);
    const lora::BgmvExpandArgs ea =
        bgmv_expand_args(token_idx, y, ldy, T, num_slices, B_slices, slice_N, slice_offset, R, L,
                         R, ranks, out, ldo, scale_expand, add_inputs, nullptr);
    if (const char *why = lora::bgmv_shrink_supported(sa)) return fail(LORA_ERR_UNSUPPORTED, "%s", why);
    if (const char *why = lora::bgmv_expand_supported(ea)) return fail(LORA_ERR_UNSUPPORTED, "%s", why);
    const lora::DeviceInfo *dev;
    if ((st = device_info(&dev)) != LORA_OK) return st;
    if (const char *why = lora::bgmv_fused_supported(sa, ea)) return fail(LORA_ERR_UNSUPPORTED, "%s", why);
    if (T == 0) return LORA_OK;
    cudaError_t e = lora::launch_bgmv_fused(dtype, sa, ea, *dev, reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? LORA_OK : cuda_fail(e, "bgmv fused shrink_expand_slice launch");
}

}  // extern "C"
