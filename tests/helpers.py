"""Shared test helpers: run a workload through the CUDA path and through the
oracle on the same seeded inputs, and compare them element by element."""
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


def f64(t: torch.Tensor) -> np.ndarray:
    return t.double().cpu().numpy()


def oracle_map(case):
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


def gpu_run_fused(lg, case, dev="cuda"):
    """plan + fused shrink/expand_slice on the GPU.  Returns (y, out, plan)."""
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
