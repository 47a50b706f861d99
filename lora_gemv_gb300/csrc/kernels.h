// Internal interface between the C ABI layer (api.cu) and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "lora_gemv.h"

namespace lora {

// Writable views of the plan arrays (see lora_plan_layout_t).
struct PlanPtrs {
    int32_t *hdr, *count, *offset, *perm, *group_lora, *group_start, *group_count;
    int4 *tiles;
    int32_t *tile_rows;  // [max_tiles][kTile]
};

struct ShrinkArgs {
    const void *x;
    int64_t ldx;
    int T, H;
    const void *A;
    int L, R, S;
    const int32_t *ranks;
    float *y;
    int64_t ldy;
    float scale;
    int add;
    int32_t *hdr;
    const int32_t *perm;
    const int4 *tiles;
    const int32_t *tile_rows;
    int max_tiles;
    int seg_plan;  // the plan was grouped from a segment table (a launch-shape hint only)
};

struct ExpandArgs {
    const float *y;
    int64_t ldy;
    int T;
    void *out;
    int64_t ldo;
    int L, R;
    const int32_t *ranks;
    int y_slice_stride;
    float scale;
    int add;
    int num_slices;
    const void *B[LORA_MAX_SLICES];
    int N[LORA_MAX_SLICES];
    int off[LORA_MAX_SLICES];
    int chunk_begin[LORA_MAX_SLICES + 1];  // first column chunk of each slice (prefix sums)
    int32_t *hdr;
    const int32_t *perm;
    const int4 *tiles;
    const int32_t *tile_rows;
    int max_tiles;
    int seg_plan;  // the plan was grouped from a segment table (a launch-shape hint only)
    int early;     // launched as the programmatic dependent of the shrink that writes y
};

// Plan-free BGMV (tokens in their natural order; every token's adapter read
// straight from the index array, or adapter 0 for all when idx is NULL).
struct BgmvShrinkArgs {
    const void *x;
    int64_t ldx;
    int T, H;
    const void *A;          // [L, S*R, H]
    int L, R, S;
    const int32_t *idx;     // [T] or NULL (every token uses adapter 0)
    const int32_t *ranks;   // [L] or NULL
    float *y;
    int64_t ldy;
    float scale;
    int add;
    int32_t *status;        // optional device word: LORA_PLANERR_TIMEOUT is OR-ed in
};

struct BgmvExpandArgs {
    const float *y;
    int64_t ldy;
    int T;
    const int32_t *idx;
    const int32_t *ranks;
    int L, R;
    int y_slice_stride;
    float scale;
    int add;
    int num_slices;
    const void *B[LORA_MAX_SLICES];
    int N[LORA_MAX_SLICES];
    int off[LORA_MAX_SLICES];
    int chunk_begin[LORA_MAX_SLICES + 1];  // first column chunk of each slice (set by the launcher)
    void *out;
    int64_t ldo;
    int32_t *status;
    // 1 when the previous kernel in the stream writes nothing the expand
    // reads but y (the chained shrink): the token indices, B and out may be
    // read before the wait for it.  0: every read waits.
    int early;
};

struct DeviceInfo {
    int sm_count;
    int max_cluster;  // largest split-K cluster the shrink kernel can be launched with
};

// 2-D fp16/bf16 tensor [rows][cols] with a row stride of `ld` elements: a TMA
// map with boxes of box_rows x 64 columns (128 bytes) in the 128-byte
// swizzled layout, zero fill outside (tmap.cu).
cudaError_t make_tensor_map_2d(CUtensorMap *m, lora_dtype_t dt, const void *base, uint64_t rows,
                               uint64_t cols, uint64_t ld, uint32_t box_rows);

cudaError_t configure_plan_kernels();
cudaError_t configure_bgmv_kernels(const DeviceInfo &dev);
cudaError_t configure_shrink_kernels(DeviceInfo *info);
cudaError_t configure_expand_kernels();

cudaError_t launch_group_tokens(const int32_t *idx, int T, int L, const PlanPtrs &p,
                                cudaStream_t stream);
cudaError_t launch_group_segments(const int32_t *ss, const int32_t *sl, const int32_t *slo, int S,
                                  int T, int L, const PlanPtrs &p, cudaStream_t stream);
// pdl: launch as a programmatic dependent of the previous kernel in the
// stream (the kernel's own griddepcontrol.wait guards every read of data the
// previous kernels produce).  Only for launches whose predecessor is known.
cudaError_t launch_shrink(lora_dtype_t dt, const ShrinkArgs &a, const DeviceInfo &dev,
                          cudaStream_t stream, bool pdl = false);
cudaError_t launch_expand(lora_dtype_t dt, const ExpandArgs &a, const DeviceInfo &dev,
                          cudaStream_t stream, bool pdl = false);

// Plan-free BGMV launches.  The *_supported checks return nullptr when the
// shape is taken, else a short reason (the caller reports LORA_ERR_UNSUPPORTED).
const char *bgmv_shrink_supported(const BgmvShrinkArgs &a);
const char *bgmv_expand_supported(const BgmvExpandArgs &a);
cudaError_t launch_bgmv_shrink(lora_dtype_t dt, const BgmvShrinkArgs &a, const DeviceInfo &dev,
                               cudaStream_t stream, bool pdl = false);
cudaError_t launch_bgmv_expand(lora_dtype_t dt, const BgmvExpandArgs &a, const DeviceInfo &dev,
                               cudaStream_t stream, bool pdl = false);

// One-launch decode pair (decode_fused.cu): a cooperative launch of clusters
// of 8 CTAs.  Takes what both halves take plus T <= 256, R <= 32, a shrink
// without add_inputs and packed y slices.
cudaError_t configure_fused_kernels(const DeviceInfo &dev);
const char *bgmv_fused_supported(const BgmvShrinkArgs &s, const BgmvExpandArgs &e);
cudaError_t launch_bgmv_fused(lora_dtype_t dt, const BgmvShrinkArgs &s, const BgmvExpandArgs &e,
                              const DeviceInfo &dev, cudaStream_t stream);

// Host-side argument checks of the C ABI (api.cu): LORA_OK or the status the
// operator would return, with lora_last_error_detail() set.
lora_status_t check_shrink(lora_dtype_t dtype, const void *x, int64_t ldx, int32_t T, int32_t H,
                           const void *A, int32_t L, int32_t R, int32_t num_slices,
                           const int32_t *ranks, const float *y, int64_t ldy, const void *plan);
lora_status_t check_expand(lora_dtype_t dtype, const float *y, int64_t ldy, int32_t T,
                           int32_t num_slices, const void *const *B_slices,
                           const int32_t *slice_N, const int32_t *slice_offset,
                           int32_t y_slice_stride, int32_t L, int32_t R, const int32_t *ranks,
                           const void *out, int64_t ldo, const void *plan);
// Returns `s` and records `msg` as this thread's lora_last_error_detail().
lora_status_t report(lora_status_t s, const char *msg);

}  // namespace lora
