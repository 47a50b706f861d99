"""Shared test helpers: run a workload through the CUDA path and through the
oracle on the same seeded inputs, and compare them element by element.

Three bounds are applied (each stated where it is defined):
* end to end, out against the oracle's out: the stated tolerance of the
  output type, |d| <= ATOL + RTOL * |ref| (TOL);
* y, the fp32 shrink output, against the oracle's y: the fp32-accumulation
  bound Y_REL * |scale| * sum_h |x[t,h] * A[l,j,h]| + Y_ABS (assert_y_fp32);
* out against the oracle's expand applied to the GPU's own y: one unit in
  the last place of the output type plus an fp32-accumulation term
  (assert_expand_ulp), so an error in the LoRA term cannot hide behind the
  looser end-to-end tolerance or the input-precision error of y.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle

# |gpu - ref| <= ATOL + RTOL * |ref|, per output dtype
TOL = {torch.float16: (1e-3, 1e-2), torch.bfloat16: (2e-3, 2e-2)}


def assert_close(got, ref, dtype, what=""):
    got = got.double().cpu().numpy() if isinstance(got, torch.Tensor) else np.asarray(got)
    ref = np.asarray(ref, np.float64)
    atol, rtol = TOL[dtype]
    err = np.abs(got - ref)
    bad = err > atol + rtol * np.abs(ref)
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError(
            f"{what}: {bad.sum()} of {bad.size} elements out of tolerance; first at {tuple(i)}: "
            f"got {got[tuple(i)]!r} ref {ref[tuple(i)]!r}; max err {err.max():.3e}")


# fp32 accumulation: products of fp16/bf16 values are exact in fp32 and every
# addition on the way to y (tensor-core K steps, stages, split-K partials)
# rounds with relative error <= 2^-23 (truncation included).  A chain of d
# additions whose rounding errors have random signs is off by about
# sqrt(d) * 2^-23 of the sum of |terms|; the deepest chain here is one CTA's
# H / 16 K steps (d = 1024 at H = 16384 without split-K: ~4e-6).  1e-5 of
# the sum of |terms| bounds that with margin (measured errors are ~1e-8 of
# it), while a y rounded to bf16 (relative error up to 2^-9 of |y|) fails it.
Y_REL, Y_ABS = 1e-5, 1e-7


def assert_y_fp32(y, case, rows=None, what=""):
    """y (GPU, fp32) against the oracle's shrink within the fp32-accumulation
    bound; the bound's sum of |terms| is the oracle's shrink of |x| and |A|."""
    lo, _, _ = oracle_map(case)
    x = case.x
    if rows is not None:
        rows = np.asarray(rows)
        lo, x = lo[rows], x[rows]
        y = y[rows]
    ranks = case.ranks.numpy() if case.ranks is not None else None
    kw = dict(num_slices=case.num_slices, ranks=ranks)
    ref = oracle.shrink(f64(x), f64(case.A), lo, scale=case.shrink_scale, **kw)
    mag = oracle.shrink(np.abs(f64(x)), np.abs(f64(case.A)), lo, scale=abs(case.shrink_scale),
                        **kw)
    got = y.double().cpu().numpy() if isinstance(y, torch.Tensor) else np.asarray(y)
    got = got[:, :ref.shape[1]]
    err = np.abs(got - ref)
    bound = Y_REL * mag + Y_ABS
    bad = err > bound
    if bad.any():
        i = tuple(np.argwhere(bad)[0])
        raise AssertionError(f"{what} y: {bad.sum()} of {bad.size} beyond the fp32 bound; first "
                             f"at {i}: got {got[i]!r} ref {ref[i]!r} bound {bound[i]:.3e}")


def ulp(v: np.ndarray, dtype) -> np.ndarray:
    """Spacing of the fp16 / bf16 numbers at |v| (subnormal spacing near 0)."""
    mant, emin = (10, -14) if dtype == torch.float16 else (7, -126)
    e = np.floor(np.log2(np.maximum(np.abs(v), 2.0 ** emin)))
    return 2.0 ** (e - mant)


# Expand feeds y to the tensor cores as a hi + lo pair of the weight type after
# a per-row power-of-two scaling (residual <= 2^-18 of the row's largest |y|
# for bf16, below fp16's subnormal spacing otherwise) and sums <= 128 products
# in fp32 (<= 128 * 2^-23); 2^-14 of sum |scale * y * B| covers both.
EXPAND_REL = 2.0 ** -14


def assert_expand_ulp(out, y, case, rows=None, what=""):
    """out (GPU) against the oracle's expand_slice of the GPU's own y: within
    one unit in the last place of the output type plus EXPAND_REL of the sum
    of |scale * y * B| (one rounding of an fp32 result, plus fp32 error)."""
    lo, _, _ = oracle_map(case)
    out0 = case.out
    if rows is not None:
        rows = np.asarray(rows)
        lo, out0 = lo[rows], out0[rows]
        y, out = y[rows], out[rows]
    ranks = case.ranks.numpy() if case.ranks is not None else None
    yd = y.double().cpu().numpy()
    Bs = [f64(b) for b in case.B]
    kw = dict(y_stride=case.R, ranks=ranks)
    ref = oracle.expand_slice(yd, Bs, case.slice_offsets, lo, f64(out0), scale=case.scale,
                              add=case.add, **kw)
    mag = oracle.expand_slice(np.abs(yd), [np.abs(b) for b in Bs], case.slice_offsets, lo,
                              np.zeros(ref.shape), scale=abs(case.scale), add=False, **kw)
    got = out.double().cpu().numpy()
    err = np.abs(got - ref)
    bound = ulp(np.maximum(np.abs(got), np.abs(ref)), case.dtype) + EXPAND_REL * mag
    bad = err > bound
    if bad.any():
        i = tuple(np.argwhere(bad)[0])
        raise AssertionError(f"{what} out: {bad.sum()} of {bad.size} beyond one ulp; first at "
                             f"{i}: got {got[i]!r} ref {ref[i]!r} bound {bound[i]:.3e}")


def f64(t: torch.Tensor) -> np.ndarray:
    return t.double().cpu().numpy()


def oracle_map(case):
    """(adapter per token, bad-id count, segment error bits) of a case; a case
    with neither token indices nor segments has every token on adapter 0."""
    if case.token_idx is None and case.seg_start is None:
        return oracle.map_tokens(np.zeros(case.T, np.int32), case.L) + (0,)
    if case.token_idx is not None:
        lo, bad = oracle.map_tokens(case.token_idx.numpy(), case.L)
        return lo, bad, 0
    return oracle.map_segments(case.seg_start.numpy(), case.seg_len.numpy(),
                               case.seg_lora.numpy(), case.T, case.L)


def gpu_plan(lg, case, dev):
    plan = lg.new_plan(case.T, case.L, dev)
    if case.token_idx is not None:
        lg.lora_group_tokens(case.token_idx.to(dev), case.L, plan)
    else:
        lg.lora_group_segments(case.seg_start.to(dev), case.seg_len.to(dev),
                               case.seg_lora.to(dev), case.T, case.L, plan)
    return plan


def gpu_run(lg, case, dev="cuda", y_in=None):
    """plan + shrink + expand_slice on the GPU.  Returns (y, out) on the host."""
    plan = gpu_plan(lg, case, dev)
    x, A = case.x.to(dev), case.A.to(dev)
    Bs = [b.to(dev) for b in case.B]
    out = case.out.to(dev)
    SR = case.num_slices * case.R
    y = torch.zeros(case.T, SR, dtype=torch.float32, device=dev) if y_in is None else y_in.to(dev)
    ranks = case.ranks.to(dev) if case.ranks is not None else None
    lg.lora_shrink(x, A, y, plan, num_slices=case.num_slices, ranks=ranks,
                   scale=case.shrink_scale, add_inputs=False)
    lg.lora_expand_slice(y, Bs, out, plan, case.slice_offsets, y_slice_stride=case.R,
                         ranks=ranks, scale=case.scale, add_inputs=case.add)
    torch.cuda.synchronize()
    return y.cpu(), out.cpu(), plan


def oracle_run(case, rows=None):
    """The oracle on all tokens, or on the token subset `rows` (tokens are
    independent, so a subset is computed exactly as in the full problem)."""
    lo, _, _ = oracle_map(case)
    x, out = case.x, case.out
    if rows is not None:
        rows = np.asarray(rows)
        lo = lo[rows]
        x, out = x[rows], out[rows]
    ranks = case.ranks.numpy() if case.ranks is not None else None
    y = oracle.shrink(f64(x), f64(case.A), lo, num_slices=case.num_slices, ranks=ranks,
                      scale=case.shrink_scale)
    o = oracle.expand_slice(y, [f64(b) for b in case.B], case.slice_offsets, lo, f64(out),
                            y_stride=case.R, ranks=ranks, scale=case.scale, add=case.add)
    return y, o


def gpu_run_chained(lg, case, dev="cuda"):
    """plan + lora_shrink_expand_slice (shrink and expand_slice chained in one
    call) on the GPU.  Returns (y, out, plan)."""
    plan = gpu_plan(lg, case, dev)
    x, A = case.x.to(dev), case.A.to(dev)
    Bs = [b.to(dev) for b in case.B]
    out = case.out.to(dev)
    y = torch.full((case.T, case.num_slices * case.R), float("nan"), dtype=torch.float32,
                   device=dev)
    ranks = case.ranks.to(dev) if case.ranks is not None else None
    lg.lora_shrink_expand_slice(x, A, y, Bs, out, plan, case.slice_offsets, ranks=ranks,
                                scale_shrink=case.shrink_scale, scale_expand=case.scale,
                                add_inputs=case.add)
    torch.cuda.synchronize()
    return y.cpu(), out.cpu(), plan
