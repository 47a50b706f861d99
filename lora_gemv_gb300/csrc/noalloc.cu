// lora_shrink_expand_slice_noalloc: the decode-path pair (BGMV grouping,
// shrink, expand_slice) for callers that cannot allocate device memory.
//
// The grouped operators read a plan (the token grouping) from a buffer the
// caller normally allocates.  Here that buffer is a fixed array in device
// global memory owned by this library: every GPU that loads the library holds
// it until the process exits.  The caller passes only inputs and outputs.
//
// Host code must not hand the array's name to a kernel: on the host it names
// a stand-in object, not device memory.  The device address is looked up once
// per device (cudaGetSymbolAddress, with that device current) and passed to
// the existing entry points as their plan pointer.
#include <stdio.h>

#include <mutex>

#include "kernels.h"

namespace {

static_assert(LORA_NOALLOC_PLAN_BYTES % 256 == 0, "whole 256-byte blocks");

// The plan of the most recent call on this device (see include/lora_gemv.h).
__device__ __align__(256) unsigned char g_noalloc_plan[LORA_NOALLOC_PLAN_BYTES];

constexpr int kMaxDevices = 64;
struct NoallocDevice {
    std::once_flag once;
    cudaError_t err = cudaSuccess;
    void *plan = nullptr;  // device address of g_noalloc_plan on this device
};
NoallocDevice g_noalloc_dev[kMaxDevices];

// Device address of the array on the current device; looked up on the first
// call made with that device current.
lora_status_t noalloc_plan(void **plan) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return lora::report(LORA_ERR_CUDA, "cudaGetDevice failed");
    if (dev < 0 || dev >= kMaxDevices) return lora::report(LORA_ERR_UNSUPPORTED, "device index");
    NoallocDevice &d = g_noalloc_dev[dev];
    std::call_once(d.once, [&] {
        d.err = cudaGetSymbolAddress(&d.plan, g_noalloc_plan);
        if (d.err != cudaSuccess) d.plan = nullptr;
    });
    if (d.err != cudaSuccess || d.plan == nullptr) {
        char msg[160];
        snprintf(msg, sizeof(msg), "cudaGetSymbolAddress of the library's plan array: %s",
                 cudaGetErrorString(d.err));
        return lora::report(LORA_ERR_CUDA, msg);
    }
    *plan = d.plan;
    return LORA_OK;
}

}  // namespace

extern "C" lora_status_t lora_shrink_expand_slice_noalloc(
    lora_dtype_t dtype, const int32_t *token_idx, const void *x, int64_t ldx, int32_t T,
    int32_t H, const void *A, int32_t L, int32_t R, const int32_t *ranks, float *y, int64_t ldy,
    int32_t num_slices, const void *const *B_slices, const int32_t *slice_N,
    const int32_t *slice_offset, void *out, int64_t ldo, float scale_shrink, float scale_expand,
    int add_inputs, lora_stream_t stream) {
    if (T > LORA_NOALLOC_MAX_TOKENS) {
        char msg[160];
        snprintf(msg, sizeof(msg), "T = %d exceeds LORA_NOALLOC_MAX_TOKENS = %d; use "
                 "lora_group_tokens with a caller-allocated plan", T, LORA_NOALLOC_MAX_TOKENS);
        return lora::report(LORA_ERR_UNSUPPORTED, msg);
    }
    lora_plan_layout_t lay;
    lora_status_t st = lora_plan_layout(T, L, &lay);
    if (st != LORA_OK) return st;
    if (lay.bytes > (int64_t)LORA_NOALLOC_PLAN_BYTES)
        return lora::report(LORA_ERR_UNSUPPORTED, "plan larger than the library's plan array");
    if (T > 0 && token_idx == nullptr) return lora::report(LORA_ERR_INVALID_ARG, "token_idx is NULL");
    void *plan = nullptr;
    if ((st = noalloc_plan(&plan)) != LORA_OK) return st;
    // every argument is checked before anything is enqueued
    st = lora::check_shrink(dtype, x, ldx, T, H, A, L, R, num_slices, ranks, y, ldy, plan);
    if (st != LORA_OK) return st;
    st = lora::check_expand(dtype, y, ldy, T, num_slices, B_slices, slice_N, slice_offset, R, L,
                            R, ranks, out, ldo, plan);
    if (st != LORA_OK) return st;
    if (T == 0) return LORA_OK;
    // The grouping kernel writes every plan word the operators read, so the
    // previous call's contents need no clearing.
    st = lora_group_tokens(token_idx, T, L, plan, (size_t)LORA_NOALLOC_PLAN_BYTES, stream);
    if (st != LORA_OK) return st;
    return lora_shrink_expand_slice(dtype, x, ldx, T, H, A, L, R, ranks, y, ldy, num_slices,
                                    B_slices, slice_N, slice_offset, out, ldo, plan, scale_shrink,
                                    scale_expand, add_inputs, stream);
}
