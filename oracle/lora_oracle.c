/*
 * Plain CPU oracle for the multi-LoRA shrink / expand / expand_slice path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product (the CUDA library and its
 * Python binding) links, imports or calls this file.  Only the tests, the
 * smoke check and the CPU-baseline leg of the benchmark use it.  It shares no
 * code, header, table or helper with the CUDA path.
 *
 * Every floating-point value arrives widened to double (fp16 / bf16 / fp32
 * widen exactly) and every sum is accumulated in double, token by token, in
 * the order the definitions below are written.  No blocking, no fusion, no
 * reordering.  OpenMP only splits the outer loop over tokens; each token's
 * arithmetic is the same serial loop whatever the thread count.
 *
 * Sources (web pages on the Punica-style multi-LoRA operators):
 *  - vLLM PR #15655 "Multi-LoRA Optimisations for the V1 TPU backend",
 *    summary list: the kernel is split into a shrink and an expand variant.
 *  - vLLM PR #11579 "Add LoRA kernel micro benchmarks": the six operators
 *    bgmv/sgmv x shrink/expand/expand_slice; add_inputs adds the group-GEMM
 *    product to the existing outputs instead of overwriting them; the expand
 *    reads an fp32 intermediate and fp16 weights (fp32 x fp16 -> fp16);
 *    m = batch x seq-len
 *    tokens, k = rank, n = hidden for expand; expand_slice writes a column
 *    slice of a fused output (num_slices).
 *  - Punica issue #17 "The smallest rank supported is 16?": BGMV gives every
 *    input its own adapter, SGMV groups inputs that share an adapter
 *    (the "AAABCC" batch) and BGMV semantics are a strict subset of SGMV's;
 *    ranks of one batch may be padded up with zeros.
 * The formulas themselves (y = x A^T into an fp32 rank buffer,
 * out[:, off:off+n] (+)= scale * y B^T, adapter index -1 = no LoRA) are the
 * operator definitions those pages name; they do not print them.
 */
#include <stdint.h>
#include <stddef.h>
#ifdef _OPENMP
#include <omp.h>
#endif

int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void oracle_set_threads(int n)
{
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/*
 * BGMV token map (Punica issue #17: every input may use a different adapter).
 * lora_of[t] = idx[t] when 0 <= idx[t] < L; -1 means "no LoRA".  Any other
 * value is counted as a bad id and treated as -1.  Returns the bad-id count.
 */
int oracle_map_tokens(const int32_t *idx, int32_t T, int32_t L, int32_t *lora_of)
{
    int bad = 0;
    for (int32_t t = 0; t < T; ++t) {
        int32_t l = idx[t];
        if (l >= 0 && l < L) {
            lora_of[t] = l;
        } else {
            if (l != -1) bad++;
            lora_of[t] = -1;
        }
    }
    return bad;
}

/*
 * SGMV token map (Punica issue #17: tokens grouped into segments that share
 * one adapter).  Segment i covers tokens [start[i], start[i] + len[i]) and
 * uses adapter lora[i].  Tokens covered by no segment get -1.
 *
 * Validity rules (the table is a list of sequences in batch order):
 *  - 0 <= start, 0 <= len, start + len <= T, else the segment is ignored and
 *    bit 1 of *err is set;
 *  - a non-empty segment must not start before the end of any earlier
 *    non-empty in-range segment (the table lists sequences in batch order),
 *    else it is ignored and bit 2 of *err is set;
 *  - lora outside [-1, L) is counted as a bad id and the segment acts as -1.
 * Returns the bad-id count.
 */
int oracle_map_segments(const int32_t *start, const int32_t *len, const int32_t *lora,
                        int32_t S, int32_t T, int32_t L, int32_t *lora_of, int32_t *err)
{
    int bad = 0;
    int64_t prev_end = 0;
    *err = 0;
    for (int32_t t = 0; t < T; ++t) lora_of[t] = -1;
    for (int32_t i = 0; i < S; ++i) {
        int64_t s0 = start[i], n = len[i];
        if (s0 < 0 || n < 0 || s0 + n > T) { *err |= 1; continue; }
        if (n == 0) continue;
        int overlaps = s0 < prev_end;
        if (s0 + n > prev_end) prev_end = s0 + n;
        if (overlaps) { *err |= 2; continue; }
        int32_t l = lora[i];
        if (!(l >= -1 && l < L)) { bad++; l = -1; }
        for (int64_t t = s0; t < s0 + n; ++t) lora_of[t] = l;
    }
    return bad;
}

/*
 * Token grouping (vLLM PR #11579's benchmark option that sorts tokens by adapter id;
 * the "AAABCC" sharing of Punica issue #17).
 *
 * by_adapter = 1 (BGMV): active tokens (lora_of >= 0) in ascending adapter
 *   id, ties kept in ascending token index (a stable sort).
 * by_adapter = 0 (SGMV): active tokens in ascending token index (segment
 *   order).
 * Then, in both cases, the inactive tokens in ascending token index.
 *
 * count[l] = number of tokens with lora_of == l; offset = exclusive prefix
 * sum of count (offset[L] = number of active tokens).
 * A group is a maximal run of equal adapter ids along perm[0 : n_active];
 * groups are then cut into tiles of at most `tile` tokens, followed by the
 * inactive tokens cut the same way with adapter -1.  tiles[4*k ..] =
 * {adapter, first perm position, token count, group number (-1 inactive)}.
 * Returns the number of tiles; *n_groups receives the number of groups.
 */
int oracle_group(const int32_t *lora_of, int32_t T, int32_t L, int by_adapter, int32_t tile,
                 int32_t *perm, int32_t *count, int32_t *offset,
                 int32_t *group_lora, int32_t *group_start, int32_t *group_count,
                 int32_t *n_groups, int32_t *tiles)
{
    for (int32_t l = 0; l < L; ++l) count[l] = 0;
    for (int32_t t = 0; t < T; ++t)
        if (lora_of[t] >= 0) count[lora_of[t]]++;
    offset[0] = 0;
    for (int32_t l = 0; l < L; ++l) offset[l + 1] = offset[l] + count[l];
    int32_t n_active = offset[L];

    int32_t pos = 0;
    if (by_adapter) {
        for (int32_t l = 0; l < L; ++l)
            for (int32_t t = 0; t < T; ++t)
                if (lora_of[t] == l) perm[pos++] = t;
    } else {
        for (int32_t t = 0; t < T; ++t)
            if (lora_of[t] >= 0) perm[pos++] = t;
    }
    for (int32_t t = 0; t < T; ++t)
        if (lora_of[t] < 0) perm[pos++] = t;

    int32_t g = 0;
    for (int32_t p = 0; p < n_active; ++p) {
        int32_t l = lora_of[perm[p]];
        if (p == 0 || l != group_lora[g - 1]) {
            group_lora[g] = l;
            group_start[g] = p;
            group_count[g] = 0;
            g++;
        }
        group_count[g - 1]++;
    }
    *n_groups = g;

    int32_t k = 0;
    for (int32_t i = 0; i < g; ++i) {
        for (int32_t p = 0; p < group_count[i]; p += tile) {
            int32_t n = group_count[i] - p < tile ? group_count[i] - p : tile;
            tiles[4 * k + 0] = group_lora[i];
            tiles[4 * k + 1] = group_start[i] + p;
            tiles[4 * k + 2] = n;
            tiles[4 * k + 3] = i;
            k++;
        }
    }
    for (int32_t p = n_active; p < T; p += tile) {
        int32_t n = T - p < tile ? T - p : tile;
        tiles[4 * k + 0] = -1;
        tiles[4 * k + 1] = p;
        tiles[4 * k + 2] = n;
        tiles[4 * k + 3] = -1;
        k++;
    }
    return k;
}

/* Rank of adapter l: ranks[l] when a rank table is given, else the stacked
 * row count R.  Values outside [0, R] are clamped (Punica issue #17: ranks
 * other than the stored one are the zero-padded rows of a larger rank). */
static int32_t rank_of(const int32_t *ranks, int32_t l, int32_t R)
{
    if (!ranks) return R;
    int32_t r = ranks[l];
    if (r < 0) r = 0;
    if (r > R) r = R;
    return r;
}

/*
 * Shrink (the "shrink" half of the split kernel in vLLM PR #15655; bgmv_shrink
 * and sgmv_shrink in vLLM PR #11579):
 *
 *   A is [L, S*R, H]: S stacked slices (q/k/v or gate/up) of R rows each.
 *   y is [T, ldy] (ldy >= S*R), kept in double here (fp32 on the GPU, per the
 *   "f32" intermediate of PR #11579's expand).
 *   For token t with adapter l = lora_of[t], slice s, row i < R, column
 *   j = s*R + i:
 *       v = scale * sum_{h < H} x[t, h] * A[l, j, h]   when l >= 0 and i < rank(l)
 *       v = 0                                          otherwise
 *       y[t, j] = (add ? y[t, j] : 0) + v
 */
void oracle_shrink(const double *x, int64_t ldx, int32_t T, int32_t H,
                   const double *A, int32_t L, int32_t R, int32_t S,
                   const int32_t *ranks, const int32_t *lora_of,
                   double scale, int add, double *y, int64_t ldy)
{
    (void)L;
#pragma omp parallel for schedule(dynamic, 4)
    for (int32_t t = 0; t < T; ++t) {
        int32_t l = lora_of[t];
        int32_t r = l >= 0 ? rank_of(ranks, l, R) : 0;
        for (int32_t s = 0; s < S; ++s) {
            for (int32_t i = 0; i < R; ++i) {
                int64_t j = (int64_t)s * R + i;
                double v = 0.0;
                if (l >= 0 && i < r) {
                    const double *a = A + ((int64_t)l * S * R + j) * H;
                    const double *xr = x + (int64_t)t * ldx;
                    double acc = 0.0;
                    for (int32_t h = 0; h < H; ++h) acc += xr[h] * a[h];
                    v = scale * acc;
                }
                double *yy = y + (int64_t)t * ldy + j;
                *yy = (add ? *yy : 0.0) + v;
            }
        }
    }
}

/*
 * Expand / expand_slice (bgmv_expand, sgmv_expand and their _slice forms in
 * vLLM PR #11579; add_inputs as discussed there):
 *
 *   Slice s has its own weights B[s] = [L, N[s], R] (row n holds the R rank
 *   coefficients of output column n), reads y columns
 *   [s*y_stride, s*y_stride + R) and writes out columns [off[s], off[s]+N[s]).
 *   For token t with adapter l = lora_of[t] and column n < N[s]:
 *       l <  0: out[t, off+n] = add ? out[t, off+n] : 0
 *       l >= 0: out[t, off+n] = (add ? out[t, off+n] : 0)
 *                               + scale * sum_{i < rank(l)} y[t, s*y_stride+i] * B[s][l, n, i]
 *   Columns outside every slice are not touched.
 *   A plain expand is the one-slice case with off = 0.
 */
void oracle_expand_slice(const double *y, int64_t ldy, int32_t T, int32_t num_slices,
                         const double *const *B, const int32_t *N, const int32_t *off,
                         int32_t y_stride, int32_t L, int32_t R, const int32_t *ranks,
                         const int32_t *lora_of, double scale, int add,
                         double *out, int64_t ldo)
{
    (void)L;
#pragma omp parallel for schedule(dynamic, 4)
    for (int32_t t = 0; t < T; ++t) {
        int32_t l = lora_of[t];
        int32_t r = l >= 0 ? rank_of(ranks, l, R) : 0;
        for (int32_t s = 0; s < num_slices; ++s) {
            for (int32_t n = 0; n < N[s]; ++n) {
                double *o = out + (int64_t)t * ldo + off[s] + n;
                if (l < 0) {
                    if (!add) *o = 0.0;
                    continue;
                }
                const double *b = B[s] + ((int64_t)l * N[s] + n) * R;
                const double *yr = y + (int64_t)t * ldy + (int64_t)s * y_stride;
                double acc = 0.0;
                for (int32_t i = 0; i < r; ++i) acc += yr[i] * b[i];
                *o = (add ? *o : 0.0) + scale * acc;
            }
        }
    }
}
