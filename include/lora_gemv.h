/*
 * lora_gemv.h - C ABI of the GB300 (sm_103a) multi-LoRA shrink / expand library.
 *
 * The operators are the Punica-style multi-LoRA pair named on these pages:
 *  - vLLM PR #15655 "[Hardware][TPU][V1] Multi-LoRA Optimisations for the V1
 *    TPU backend", summary list: the LoRA kernel is split into a shrink and
 *    an expand variant, with block skipping and fast mask creation;
 *  - vLLM PR #11579 "[misc] Add LoRA kernel micro benchmarks": the operators
 *    bgmv_shrink, bgmv_expand, bgmv_expand_slice, sgmv_shrink, sgmv_expand,
 *    sgmv_expand_slice; the add_inputs flag of expand (the product is added
 *    to out); the fp32 intermediate between shrink and expand (fp32 times
 *    fp16 weights giving fp16); the
 *    num_slices of a fused output; split-K shrink that adds partials;
 *  - Punica issue #17 "The smallest rank supported is 16?": BGMV (one adapter
 *    per input) versus SGMV (segments of inputs sharing one adapter, the
 *    "AAABCC" batch), BGMV semantics being a subset of SGMV's, and ranks
 *    padded up to a common size as the old workaround.
 *
 * Definitions (T tokens, H hidden size, L stacked adapters, R rows per slice
 * = the largest rank, r_l = rank of adapter l <= R, l = adapter of token t,
 * l = -1 meaning "no LoRA"):
 *   shrink : y[t, s*R + i] = (add ? y[t, s*R+i] : 0) + scale * sum_h x[t,h] * A[l, s*R+i, h]
 *            for i < r_l; the term is 0 for i >= r_l and for l = -1.
 *   expand : out[t, off_s + n] = (add ? out[t, off_s+n] : 0)
 *                               + scale * sum_{i<r_l} y[t, s*ys + i] * B_s[l, n, i]
 *            for l >= 0; for l = -1 the row is left untouched (add) or set to 0.
 *   BGMV and SGMV differ only in how the token -> adapter map is given; both
 *   are turned into one "plan" (token grouping) that every operator reads.
 *
 * Conventions
 *  - Every pointer argument named x, A, B*, y, out, plan, token_idx, seg_*,
 *    ranks is a DEVICE pointer on the current CUDA device; host arrays are
 *    marked "host".  The caller owns all memory.  The library allocates no
 *    device or host memory, keeps no per-call state and never synchronises
 *    inside an operator: each operator only enqueues kernels on `stream`,
 *    so the calls may be captured in a CUDA graph.
 *  - Matrices are row-major with an explicit leading dimension (in elements).
 *  - fp16 / bf16 elements are IEEE binary16 / bfloat16; y is fp32.
 *  - Arithmetic: products of fp16/bf16 values accumulated in fp32 on tensor
 *    cores; expand feeds y to the tensor cores as a hi+lo pair of the weight
 *    type scaled per token row by a power of two, so y keeps ~fp32 accuracy;
 *    the result is rounded once (round-to-nearest-even) to the output type.
 *    Summation order is not specified: results agree with an exact sum to
 *    fp32-accumulation accuracy, not bit-for-bit across launch shapes.
 *  - Errors: argument errors are detected on the host, before anything is
 *    enqueued, and returned synchronously; nothing is launched then.  A
 *    failed launch returns LORA_ERR_CUDA.  Conditions only visible on the
 *    device (bad adapter ids, a malformed segment table, a plan that does not
 *    match the operator's T / L) are recorded in the plan's error words and
 *    read back with lora_get_error(); the kernels never trap or spin.
 *  - Thread safety: all functions are re-entrant.  The first call on a
 *    device configures kernel attributes once (guarded); make that first
 *    call outside stream capture.
 */
#ifndef LORA_GEMV_H
#define LORA_GEMV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A cudaStream_t (the CUDA runtime's stream handle); NULL = legacy default stream. */
typedef struct CUstream_st *lora_stream_t;

typedef enum {
    LORA_OK = 0,
    LORA_ERR_INVALID_ARG = 1, /* a size, stride, pointer or flag is out of its documented range */
    LORA_ERR_UNSUPPORTED = 2, /* valid but outside this build's limits (e.g. L > LORA_MAX_ADAPTERS) */
    LORA_ERR_WORKSPACE = 3,   /* plan buffer too small or misaligned */
    LORA_ERR_CUDA = 4         /* the CUDA runtime reported an error (launch, attribute, device query) */
} lora_status_t;

typedef enum { LORA_F16 = 0, LORA_BF16 = 1 } lora_dtype_t;

#define LORA_TILE_TOKENS 64      /* tokens per work tile of the plan */
#define LORA_MAX_RANK 128        /* largest R (rows per slice / max adapter rank) */
#define LORA_MAX_SLICES 8        /* largest num_slices of shrink / expand_slice */
#define LORA_MAX_ADAPTERS 1024   /* largest L accepted by lora_group_tokens */
#define LORA_MAX_TOKENS (1 << 24)

/* Plan header words (int32, at byte offset 0 of the plan). */
enum {
    LORA_HDR_MAGIC = 0,    /* LORA_PLAN_MAGIC once a grouping call has run */
    LORA_HDR_T = 1,
    LORA_HDR_L = 2,
    LORA_HDR_KIND = 3,     /* 1 = built from token indices (BGMV), 2 = from segments (SGMV) */
    LORA_HDR_NACTIVE = 4,  /* tokens with an adapter */
    LORA_HDR_NGROUPS = 5,
    LORA_HDR_NTILES = 6,
    LORA_HDR_BAD_IDS = 7,  /* adapter ids outside [-1, L): treated as -1 */
    LORA_HDR_ERR = 8,      /* LORA_PLANERR_* bits, OR-ed by grouping and by operators */
    LORA_HDR_WORDS = 16
};
#define LORA_PLAN_MAGIC 0x4C6F5241
#define LORA_PLANERR_SEG_RANGE 1    /* a segment had start < 0, len < 0 or start+len > T: ignored */
#define LORA_PLANERR_SEG_ORDER 2    /* a segment began before the end of an earlier one: ignored */
#define LORA_PLANERR_MISMATCH 4     /* an operator got a plan built for another T or L: it wrote nothing */
#define LORA_PLANERR_TIMEOUT 8      /* a kernel's bounded wait for its cluster peers expired: its
                                       outputs for that call are not valid (never expected) */
#define LORA_PLANERR_BOUNDS 16      /* LORA_DEBUG builds only: a plan entry read by an operator was
                                       outside its range (a token row outside [-1, T), an adapter
                                       id outside [-1, L), a tile row count outside [0, 64]).
                                       Every build skips such entries (the row or the tile gets no
                                       term); debug builds also count them here. */

/*
 * Plan layout: byte offsets of each array inside the caller's plan buffer.
 * The layout depends only on (T, L).
 *   count[L]          tokens per adapter
 *   offset[L+1]       exclusive prefix sum of count (BGMV: where adapter l's
 *                     tokens start in perm)
 *   perm[T]           token order: perm[0:n_active] = tokens with an adapter,
 *                     grouped (BGMV: ascending adapter id, ties by token index;
 *                     SGMV: ascending token index), then the tokens without
 *                     an adapter in ascending order
 *   group_lora/start/count[T+1]  maximal runs of one adapter along
 *                     perm[0:n_active]: adapter id, first perm position, length
 *   tiles[max_tiles][4]  each group cut into pieces of <= LORA_TILE_TOKENS
 *                     tokens, then the inactive tokens likewise:
 *                     {adapter (-1 for inactive), first perm position,
 *                      token count, group number (-1 for inactive)}
 *   tile_rows[max_tiles][LORA_TILE_TOKENS]  the tokens of each tile
 *                     (perm[first .. first + count)), -1 past the count, so
 *                     an operator reads a tile's rows without first reading
 *                     its record
 */
typedef struct {
    int64_t header, count, offset, perm, group_lora, group_start, group_count, tiles, tile_rows;
    int64_t max_tiles;
    int64_t bytes; /* total size of the buffer */
} lora_plan_layout_t;

/* Fills *layout for a plan of T tokens and L adapters.
 * Errors: LORA_ERR_INVALID_ARG (T < 0, L < 1, layout NULL), LORA_ERR_UNSUPPORTED
 * (T > LORA_MAX_TOKENS). */
lora_status_t lora_plan_layout(int32_t T, int32_t L, lora_plan_layout_t *layout);

/* Size in bytes of the plan buffer for (T, L); 0 on invalid arguments.  The
 * buffer must be 16-byte aligned device memory. */
size_t lora_workspace_size(int32_t T, int32_t L);

/*
 * BGMV grouping (Punica issue #17: every input may use its own adapter;
 * vLLM PR #15655 summary: cheap mask construction): builds the plan from a per-token
 * adapter index token_idx[T] (device, int32; -1 = no LoRA; other values
 * outside [0, L) are counted in LORA_HDR_BAD_IDS and treated as -1).
 * One single-block kernel on `stream`; the grouping is a stable counting sort.
 * Errors: LORA_ERR_INVALID_ARG (NULL pointers with T > 0, T < 0, L < 1),
 * LORA_ERR_UNSUPPORTED (L > LORA_MAX_ADAPTERS, T > LORA_MAX_TOKENS),
 * LORA_ERR_WORKSPACE (plan_bytes < lora_workspace_size(T, L) or plan not
 * 16-byte aligned), LORA_ERR_CUDA.
 */
lora_status_t lora_group_tokens(const int32_t *token_idx, int32_t T, int32_t L,
                                void *plan, size_t plan_bytes, lora_stream_t stream);

/*
 * SGMV grouping (Punica issue #17: inputs grouped into segments sharing an
 * adapter; vLLM PR #11579's seq-len / sort-by-lora-id): builds the plan from
 * a segment table of num_segs entries (device, int32 each):
 * segment i covers tokens [seg_start[i], seg_start[i] + seg_len[i]) with
 * adapter seg_lora[i].  Tokens covered by no segment, and segments with
 * adapter -1, get no LoRA.  A segment with start < 0, len < 0 or
 * start + len > T is ignored (LORA_PLANERR_SEG_RANGE); a non-empty segment
 * that starts before the end of an earlier non-empty in-range segment is
 * ignored (LORA_PLANERR_SEG_ORDER); adapter ids outside [-1, L) count as bad
 * ids and act as -1.  Adjacent runs of one adapter are coalesced into one
 * group.  One single-block kernel on `stream`.
 * Errors: as lora_group_tokens (num_segs < 0 is LORA_ERR_INVALID_ARG).
 */
lora_status_t lora_group_segments(const int32_t *seg_start, const int32_t *seg_len,
                                  const int32_t *seg_lora, int32_t num_segs, int32_t T,
                                  int32_t L, void *plan, size_t plan_bytes,
                                  lora_stream_t stream);

/*
 * Shrink (bgmv_shrink / sgmv_shrink; vLLM PR #11579, split-K shrink note):
 *   x    [T, ldx]       activations, dtype `dtype` (ldx >= H)
 *   A    [L, S*R, H]    stacked adapters, contiguous; S = num_slices slices
 *                       (q/k/v or gate/up) of R rows each; rows i >= r_l of a
 *                       slice are never read
 *   ranks [L] or NULL   per-adapter rank r_l (device int32, clamped to [0, R]);
 *                       NULL means every adapter has rank R
 *   y    [T, ldy] fp32  output (ldy >= S*R); every column j < S*R of every
 *                       row is written (add = 0) or accumulated (add != 0);
 *                       columns >= S*R are not touched
 *   plan                from lora_group_tokens / lora_group_segments with
 *                       the same T and L
 * Limits: 1 <= R <= LORA_MAX_RANK, 1 <= num_slices <= LORA_MAX_SLICES,
 * H >= 1.  T == 0 launches nothing (x and y may then be NULL).
 * Errors: LORA_ERR_INVALID_ARG (NULL pointers, bad sizes or strides, bad
 * dtype), LORA_ERR_UNSUPPORTED, LORA_ERR_CUDA.
 */
lora_status_t lora_shrink(lora_dtype_t dtype, const void *x, int64_t ldx, int32_t T, int32_t H,
                          const void *A, int32_t L, int32_t R, int32_t num_slices,
                          const int32_t *ranks, float *y, int64_t ldy, const void *plan,
                          float scale, int add_inputs, lora_stream_t stream);

/*
 * Expand (bgmv_expand / sgmv_expand; add_inputs as in vLLM PR #11579):
 *   y    [T, ldy] fp32  the shrink output, columns [0, R) read (r_l of them)
 *   B    [L, N, R]      adapters, contiguous; column i >= r_l never read
 *   out  [T, ldo]       dtype `dtype`; columns [0, N) of active tokens are
 *                       updated; rows of tokens without an adapter are left
 *                       untouched (add != 0) or zeroed (add == 0)
 * Equivalent to lora_expand_slice with one slice at offset 0.
 * Errors: as lora_expand_slice.
 */
lora_status_t lora_expand(lora_dtype_t dtype, const float *y, int64_t ldy, int32_t T,
                          const void *B, int32_t L, int32_t N, int32_t R, const int32_t *ranks,
                          void *out, int64_t ldo, const void *plan, float scale, int add_inputs,
                          lora_stream_t stream);

/*
 * Expand into column slices of a fused output (bgmv_expand_slice /
 * sgmv_expand_slice; vLLM PR #11579 num_slices), all slices in one launch:
 *   B_slices   host array of num_slices device pointers, slice s is [L, N_s, R]
 *   slice_N    host array, N_s >= 0
 *   slice_offset host array, first out column of slice s; the slices' column
 *              ranges must not overlap and must lie inside [0, ldo)
 *   y_slice_stride  slice s reads y columns [s*y_slice_stride, s*y_slice_stride + R)
 *              (R for a y produced by a stacked shrink); must keep them inside ldy
 *   out columns outside every slice are never read or written.
 *   T == 0 launches nothing (y and out may then be NULL).
 * Errors: LORA_ERR_INVALID_ARG (NULL pointers, overlapping or out-of-range
 * slices, bad strides, bad dtype), LORA_ERR_UNSUPPORTED, LORA_ERR_CUDA.
 */
lora_status_t lora_expand_slice(lora_dtype_t dtype, const float *y, int64_t ldy, int32_t T,
                                int32_t num_slices, const void *const *B_slices,
                                const int32_t *slice_N, const int32_t *slice_offset,
                                int32_t y_slice_stride, int32_t L, int32_t R,
                                const int32_t *ranks, void *out, int64_t ldo, const void *plan,
                                float scale, int add_inputs, lora_stream_t stream);

/*
 * Shrink followed by expand_slice in one call (vLLM PR #15655's shrink and
 * expand variants of the LoRA kernel, chained through the fp32 rank buffer
 * of vLLM PR #11579), the decode-path form used once per LoRA layer:
 *   y   = scale_shrink * x . A[l]^T         (as lora_shrink with add_inputs = 0,
 *                                             A = [L, num_slices*R, H])
 *   out = (add_inputs ? out : 0) + scale_expand * y_s . B_s[l]^T for every slice
 *                                            (as lora_expand_slice with y_slice_stride = R)
 * y [T, ldy >= num_slices*R] is written in full (it is also the fp32 output of
 * the shrink).  The two kernels are chained with programmatic dependent
 * launch: the expand starts while the shrink finishes, reading the plan, out
 * and B_s early and y only once the shrink's results are visible, so the
 * pair costs close to one launch.  Results are those of the two-operator
 * sequence.
 * Errors: those of lora_shrink and lora_expand_slice.
 */
lora_status_t lora_shrink_expand_slice(lora_dtype_t dtype, const void *x, int64_t ldx, int32_t T,
                                       int32_t H, const void *A, int32_t L, int32_t R,
                                       const int32_t *ranks, float *y, int64_t ldy,
                                       int32_t num_slices, const void *const *B_slices,
                                       const int32_t *slice_N, const int32_t *slice_offset,
                                       void *out, int64_t ldo, const void *plan,
                                       float scale_shrink, float scale_expand, int add_inputs,
                                       lora_stream_t stream);

/*
 * Plan-free BGMV (bgmv_shrink / bgmv_expand_slice of vLLM PR #11579; the
 * per-input adapter of Punica issue #17; the mask-free single-adapter path
 * and the skipping of blocks without work of vLLM PR #15655's summary list).
 *
 * The decode-path form for batches served by a few adapters: no plan and no
 * grouping launch.  Tokens stay in their natural order; each block of 128
 * consecutive tokens is contracted against the weights of every adapter that
 * has a token in it, and each token keeps its own adapter's result.  The
 * definitions, the meaning of y, ranks, slices, scale and add_inputs, and the
 * results (to fp32-accumulation accuracy) are those of the grouped operators
 * above with the plan of lora_group_tokens(token_idx).
 *
 *   token_idx [T]  device int32 adapter index per token (-1 = no LoRA; other
 *                  values outside [0, L) also act as -1, and are not counted:
 *                  lora_group_tokens counts them).  NULL means every token
 *                  uses adapter 0: the dense single-adapter case, with no
 *                  index read and no masking.
 *   status         optional device int32 (NULL = none): LORA_PLANERR_TIMEOUT is
 *                  OR-ed into it if a kernel's bounded wait expired (never
 *                  expected; that call's outputs are then not valid).
 *
 * Shapes taken (LORA_ERR_UNSUPPORTED otherwise, before anything is enqueued;
 * the grouped operators take every shape):
 *   L <= LORA_BGMV_MAX_ADAPTERS, T <= LORA_BGMV_MAX_TOKENS;
 *   shrink: x and A 16-byte aligned, ldx and H multiples of 8,
 *           num_slices * R a multiple of 8;
 *   expand: R a multiple of 8 and <= 64, L * (R rounded up to 16) <= 128,
 *           y 16-byte aligned with ldy and y_slice_stride multiples of 4,
 *           out 16-byte aligned with ldo, every slice width and offset
 *           multiples of 8, every B_s 16-byte aligned.
 * With a rank table, rows / columns >= r_l are never used in the result (the
 * shrink reads A rows up to R and discards the extra products).
 * For R > 32 or T > 256 the expand writes out back in 64-column tiles of 128
 * token rows: with add_inputs, the rows of tokens without a LoRA term are
 * rewritten with the values just read (their contents do not change, but out
 * must not be written concurrently by other work); without add_inputs they
 * become zero.  For R <= 32 and T <= 256 (the fp32 FMA expand) those rows
 * are left alone with add_inputs.
 * Columns outside the slices are never written.
 * Errors: as the grouped operators (no plan argument), plus
 * LORA_ERR_UNSUPPORTED for shapes outside the list above.
 */
#define LORA_BGMV_MAX_ADAPTERS 8
#define LORA_BGMV_MAX_TOKENS (65535 * 128)
lora_status_t lora_bgmv_shrink(lora_dtype_t dtype, const int32_t *token_idx, const void *x,
                               int64_t ldx, int32_t T, int32_t H, const void *A, int32_t L,
                               int32_t R, int32_t num_slices, const int32_t *ranks, float *y,
                               int64_t ldy, float scale, int add_inputs, int32_t *status,
                               lora_stream_t stream);

lora_status_t lora_bgmv_expand_slice(lora_dtype_t dtype, const int32_t *token_idx, const float *y,
                                     int64_t ldy, int32_t T, int32_t num_slices,
                                     const void *const *B_slices, const int32_t *slice_N,
                                     const int32_t *slice_offset, int32_t y_slice_stride,
                                     int32_t L, int32_t R, const int32_t *ranks, void *out,
                                     int64_t ldo, float scale, int add_inputs, int32_t *status,
                                     lora_stream_t stream);

/* Shrink then expand_slice (y_slice_stride = R), the expand chained to the
 * shrink by programmatic dependent launch: it stages its out tiles and B rows
 * while the shrink runs and reads y once the shrink grid has completed. */
lora_status_t lora_bgmv_shrink_expand_slice(lora_dtype_t dtype, const int32_t *token_idx,
                                            const void *x, int64_t ldx, int32_t T, int32_t H,
                                            const void *A, int32_t L, int32_t R,
                                            const int32_t *ranks, float *y, int64_t ldy,
                                            int32_t num_slices, const void *const *B_slices,
                                            const int32_t *slice_N, const int32_t *slice_offset,
                                            void *out, int64_t ldo, float scale_shrink,
                                            float scale_expand, int add_inputs, int32_t *status,
                                            lora_stream_t stream);

/*
 * The same result as lora_bgmv_shrink_expand_slice (y included) from ONE
 * kernel launch: a cooperative launch of clusters of 8 CTAs (at most one CTA
 * per SM) in two phases separated by a grid-wide barrier.  Phase one: the
 * shrink, one (adapter, slice) per cluster, K split over the cluster's CTAs
 * and the partial products added in distributed shared memory in a fixed
 * order; phase two: the expand.  It answers the fixed cost of the two
 * launches a decode step otherwise pays per layer, the cost the split into
 * shrink and expand kernels brings (vLLM PR #15655, the summary list).
 *
 * Arguments, layouts and ownership are those of lora_bgmv_shrink_expand_slice
 * (there is no status word: the kernel has no bounded waits).  Shapes taken,
 * in addition to those of the two halves: T <= LORA_FUSED_MAX_TOKENS,
 * R <= 32.  y and out do not change from run to run and stay within the
 * bounds of the two-launch form.  With add_inputs, rows without a LoRA term
 * are never written.
 * Errors: as lora_bgmv_shrink_expand_slice, plus LORA_ERR_UNSUPPORTED for
 * shapes outside the list and on devices where the kernel's clusters do not
 * fit; LORA_ERR_CUDA if the cooperative launch is refused.
 */
#define LORA_FUSED_MAX_TOKENS 256
lora_status_t lora_bgmv_fused_shrink_expand_slice(
    lora_dtype_t dtype, const int32_t *token_idx, const void *x, int64_t ldx, int32_t T, int32_t H,
    const void *A, int32_t L, int32_t R, const int32_t *ranks, float *y, int64_t ldy,
    int32_t num_slices, const void *const *B_slices, const int32_t *slice_N,
    const int32_t *slice_offset, void *out, int64_t ldo, float scale_shrink, float scale_expand,
    int add_inputs, lora_stream_t stream);

/*
 * lora_shrink_expand_slice for callers that cannot allocate device memory.
 * The pages have no counterpart of this entry point: it is a convenience of
 * this library, not a step of the method.
 *
 * Who needs it: a caller that receives its input and output buffers from a
 * host that owns all device memory (a plugin's enqueue step in an inference
 * engine, for example) has no way to obtain the plan buffer the other
 * entry points require, and a latency-critical serving loop may not accept
 * cudaMalloc, which can synchronise the device.  This call needs only the
 * inputs and outputs: it groups token_idx (as lora_group_tokens) into a plan
 * kept in a fixed device array owned by the library, then runs
 * lora_shrink_expand_slice on that plan.  It calls no cudaMalloc, cudaFree or
 * other allocating routine.
 *
 * Arguments: those of lora_shrink_expand_slice, with token_idx [T] (device,
 * int32, the BGMV adapter index of each token; -1 = no LoRA; values outside
 * [-1, L) count as bad ids and act as -1) in place of the plan.  Results are
 * those of lora_group_tokens followed by lora_shrink_expand_slice.
 *
 * Limits: T <= LORA_NOALLOC_MAX_TOKENS (4096); larger T returns
 * LORA_ERR_UNSUPPORTED before anything is enqueued.  The array is
 * LORA_NOALLOC_PLAN_BYTES (1.25 MiB) of device memory on every GPU that
 * loads the library, held until the process exits.
 *
 * Set-up: the first call made with a given device current looks up the
 * array's device address on that device (cudaGetSymbolAddress); make that
 * first call before any stream capture.
 *
 * Shared state: every call on a device uses the same array and leaves its
 * plan there (nothing in it has to start at zero: each call's grouping
 * rewrites every word its operators read).  Calls whose work overlaps on the
 * GPU (other streams, other threads, unordered graph branches) race on the
 * array and may produce wrong results; order them, e.g. on one stream.  The
 * plan's error words are not readable through this entry point.
 * Errors: those of lora_group_tokens and lora_shrink_expand_slice, plus
 * LORA_ERR_UNSUPPORTED for T > LORA_NOALLOC_MAX_TOKENS and LORA_ERR_CUDA if
 * the array's address cannot be obtained.
 */
#define LORA_NOALLOC_MAX_TOKENS 4096
#define LORA_NOALLOC_PLAN_BYTES (1280 * 1024)
lora_status_t lora_shrink_expand_slice_noalloc(lora_dtype_t dtype, const int32_t *token_idx,
                                               const void *x, int64_t ldx, int32_t T, int32_t H,
                                               const void *A, int32_t L, int32_t R,
                                               const int32_t *ranks, float *y, int64_t ldy,
                                               int32_t num_slices, const void *const *B_slices,
                                               const int32_t *slice_N,
                                               const int32_t *slice_offset, void *out,
                                               int64_t ldo, float scale_shrink,
                                               float scale_expand, int add_inputs,
                                               lora_stream_t stream);

/*
 * Reads the plan's device-side error words.  SYNCHRONISES `stream` (a
 * device-to-host copy); for tests and debugging, not for the hot path.
 * *bad_ids <- LORA_HDR_BAD_IDS, *err_flags <- LORA_HDR_ERR (either may be NULL).
 * Errors: LORA_ERR_INVALID_ARG (plan NULL), LORA_ERR_CUDA.
 */
lora_status_t lora_get_error(const void *plan, int32_t *bad_ids, int32_t *err_flags,
                             lora_stream_t stream);

/* Static description of a status code. */
const char *lora_status_string(lora_status_t status);

/* Thread-local text describing the last non-OK status returned on this thread. */
const char *lora_last_error_detail(void);

/* Library ABI version (major * 10000 + minor * 100 + patch). */
int32_t lora_version(void);

#ifdef __cplusplus
}
#endif
#endif /* LORA_GEMV_H */
